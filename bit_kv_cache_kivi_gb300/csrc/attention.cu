// attention.cu -- decode attention over the packed KIVI cache.
//
// Decode step 2 of the chooblog KIVI review (§1.3): A = softmax(t_Q X_K^T),
// t_O = A X_V, scaled by 1/sqrt(D) as in the notebook "KIVI - 2-bit KV cache
// quantisation"; dequantization is fused into both products (review §3.2
// "System-Level": no separate dequantize pass).
//
// The context is split along the tokens (flash-decoding).  Split 0 of every
// (batch, kv-head, head chunk) takes the tail [t_tail, l) -- the tokens whose
// keys or values are still fp16 in the residual rings, plus the partial value
// group before them -- on CUDA cores.  Splits 1.. take the fully packed
// 32-token tiles [0, t_tail).  Partials are merged in the same launch: the
// CTA that finishes last in a group of up to kMergeGroup splits merges the
// group, and with more than one group the last group merges the groups;
// nothing ever waits on another CTA.
//
// Packed tiles (2, 3, 4 or 8 bits) run on the tensor cores (mma.sync
// m16n8k16, fp16 operands, fp32 accumulation).  Each warp streams its tiles
// through its own ring of staged tiles (one lane issues one bulk copy per
// tile, completion on an mbarrier) and keeps an online softmax per head:
//   scores  S[t, j] = sum_d c_td (q_jd s_d) + beta_j, beta_j = sum_d q_jd z_d
//   output  O[d, j] = sum_t c_td (p_jt s_t,g(d)) + sum_t p_jt z_t,g(d)
// The codes c enter the MMA as fp16 subnormals c * base^i * 2^-24 (the masked
// code bits are the whole encoding; base 4 at 2 and 3 bits, 16 at 4, 1 at 8);
// the fp32 factors q*s and p*s enter as an
// fp16 hi/lo pair (hi = fp16(x), lo = fp16(x - hi)) in the 8 columns of the
// n=8 operand as (head, hi) and (head, lo): four query heads per MMA, and the
// sum hi + lo recovers x to about 2^-22.  Each query head is first scaled by a
// power of two so that max |q| < 1, and a head's running max trails its
// scores by at most 0.5 (log2 units), so neither q*s nor p*s can overflow
// fp16.
#include <cuda_bf16.h>

#include <cstddef>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;
constexpr int kNH = kHeadChunk;  // query heads per CTA (one "head chunk")
// A bounded wait for staged data gives up after this long (the copies take
// microseconds); the CTA then records the failure in the status word.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

__device__ __forceinline__ float load_q(const void* q, long idx, int dt) {
  if (dt == kF32) return static_cast<const float*>(q)[idx];
  if (dt == kF16) return __half2float(static_cast<const __half*>(q)[idx]);
  return __uint_as_float((uint32_t)static_cast<const uint16_t*>(q)[idx] << 16);
}

__device__ __forceinline__ float h_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}

__device__ __forceinline__ float h_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// fp16x2 arithmetic on raw 32-bit registers (round to nearest even).
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// {lo, hi} floats -> fp16x2 (nearest even); the first argument is the low half.
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// a * b - c in fp16x2 (one rounding; the negation folds into the FMA)
__device__ __forceinline__ uint32_t hfms2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("{\n\t.reg .b32 nc;\n\tneg.f16x2 nc, %3;\n\tfma.rn.f16x2 %0, %1, %2, nc;\n}"
      : "=r"(d)
      : "r"(a), "r"(b), "r"(c));
  return d;
}

// x * s for an fp32 x given as an fp16 pair (xa, xb) with x = xa + xb, split
// again as hi + lo across lanes: a "hi" lane passes (xa = hi(x), xb = 0) and
// gets fp16(x * s); a "lo" lane passes (xa = lo(x), xb = hi(x)) and gets
// fp16(xa * s + (xb * s - fp16(xb * s))), the residual of the hi product being
// exact in fp16.  Three fp16x2 instructions, no select.
__device__ __forceinline__ uint32_t split_mul(uint32_t xa, uint32_t xb, uint32_t s) {
  return hfma2u(xa, s, hfms2u(xb, s, hmul2u(xb, s)));
}

// Value rows are group-interleaved: the byte unit of channels 32*gp + 4*w ..
// +3 sits at unit position 4*w + gp (units are bits/2 bytes).
__device__ __forceinline__ int v_unit_pos(int unit) { return 4 * (unit & 7) + (unit >> 3); }

// v[i] for a lane-dependent i without dynamic register indexing.
__device__ __forceinline__ float pick4(const float (&v)[4], int i) {
  float r = v[0];
  r = i == 1 ? v[1] : r;
  r = i == 2 ? v[2] : r;
  r = i == 3 ? v[3] : r;
  return r;
}

// ---------------------------------------------------------------------------
// Shared memory.

// q tables in MMA fragment order.  Lane (g, tig) reads the 16 words of
// column g (head g >> 1, part g & 1) for its tig, as four 16-byte quarters;
// the layout [quarter][column][tig] spreads the 8 lanes of a shared-memory
// phase over distinct banks.  Word w (k-step ks = w >> 1) of (column, tig)
// holds the channel pair of code position i:
//   2 bits: word m = tig + 4*(ks >> 2) of a key row, i = 2*(ks & 3) + (w & 1),
//           channels (16m + i, 16m + i + 8);
//   4 bits: word m = tig + 4*(ks >> 1), i = 2*(ks & 1) + (w & 1),
//           channels (8m + i, 8m + i + 4).
//
// A staged packed tile keeps the cache's own layouts (one bulk copy per
// array): codes as (16 * BITS)-byte rows, key scales / zeros as fp16 [128],
// value scales / zeros as fp16 [32 tokens][4 groups].
template <int BITS>
struct TileBuf {
  uint32_t kc[128 * BITS];                // key codes
  uint32_t vc[128 * BITS];                // value codes (group-interleaved rows)
  uint32_t sk[64], zk[64];
  uint32_t sv[64], zv[64];
  uint32_t outl[outlier_block_bytes(kMaxOutliers) / 4];  // outlier block, when the cache keeps outliers
};
template <int BITS>
constexpr int kStagesOf = BITS == 2 ? 3 : 2;  // tiles in flight per warp (3 KB / 4-9 KB tiles)

template <int BITS>
struct WarpSmem {
  TileBuf<BITS> st[kWarps][kStagesOf<BITS>];  // per-warp rings of staged tiles
  uint4 qs[2][4][8][4];                   // q * base^-e(i) as split_mul operands (xa, xb)
  uint4 qb[4][8][4];                      // q hi / lo
  float pbuf[kWarps][kNH][34];            // one tile's weights per warp, token order
                                          // 8 (t & 3) + 4 (t >> 4) + 2 ((t >> 3) & 1) + ((t >> 2) & 1)
  float qv[kNH][kHeadDim];                // q, staged for the tables
  float qscale[kNH];                      // 2^E_j * softmax scale * log2(e)
  int qexp[kNH];                          // E_j: max |q_j| * 2^-E_j lies in [0.5, 1)
  unsigned long long bar[kWarps][kStagesOf<BITS>];
};

// A tail split: up to kTailTok tokens, each staged as a 256-byte key row and
// a 256-byte value row -- an fp16 residual row (16-byte chunks XOR-swizzled by
// row), or the packed codes at the row start; the scale / zero blocks of the
// packed tiles involved are staged whole (kg, vg), in the tiles' order.
static_assert(kNH == 4, "the tail split keeps the heads of a channel / token in one float4");
struct TailSmem {
  float4 q4[kHeadDim];                    // q * scale * log2(e): the kNH heads of channel d
  uint4 krow[kTailTok][16];
  uint4 vrow[kTailTok][16];
  uint32_t kg[2][2][64];                  // scale / zero of the (at most two) key groups
  uint32_t ko[2][outlier_block_bytes(kMaxOutliers) / 4];  // their outlier blocks
  uint32_t vg[2][2][64];                  // value scale / zero blocks of the (at most two) tiles
  float4 p4[kTailTok];                    // per token: scores, then weights, of the kNH heads
  float mh[kNH], lh[kNH];                 // per head: max and sum of the weights
};

template <int BITS>
union SplitSmem {
  WarpSmem<BITS> ws;
  TailSmem tail;
};

enum Path { kPathMma = 1, kPathTail = 2 };

// Per-warp merge area: [kNH][kHeadDim] floats inside buffers that the CTA
// is done with (its staged tiles or tail rows).
template <int BITS>
__device__ __forceinline__ float* merge_area(SplitSmem<BITS>& sm, int warp, int path) {
  if (path == kPathMma) return reinterpret_cast<float*>(&sm.ws.st[warp][0]);
  return reinterpret_cast<float*>(&sm.tail.krow[0][0]) + warp * kNH * kHeadDim;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// mbarrier + bulk copy (one elected thread issues; the barrier's transaction
// count completes the phase when every byte has landed).
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the completion of phase `parity` of an mbarrier, for at most
// kWaitLimitNs.  Returns false on timeout.
__device__ __noinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Diagnostics: one thread waits, with the bounded wait above, on phase 0 of
// an mbarrier that nothing completes (no copy is issued, no thread arrives),
// and records the timeout in *status as a packed split does in the
// workspace status word.
__global__ void wait_probe_kernel(int* status) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (!mbar_wait(&bar, 0u)) atomicOr(status, 1);
  }
}

// ---------------------------------------------------------------------------
// A tail split on CUDA cores: tokens [c0, c0 + n), n <= kTailTok, of the tail
// [t_tail, l), staged in one round of copies (fp16 residual rows, packed rows
// and the key groups' scales / zeros); then scores with four threads per
// token (32 channels each), the softmax of a head per warp, and the value sum
// with one thread per channel.  Keys and values of packed rows are
// dequantized as c * s + z with a single rounding, which equals the
// notebook's fl(fl(c * s) + z) because c * s is exact in fp32.  Leaves the
// partial of the CTA in warp 0's slots (the other warps' slots empty).
template <int BITS>
__device__ void tail_split(const CacheView& cv, const AttnArgs& a, const SeqPlan p, SplitSmem<BITS>& sm,
                           long unit, int b,
                           int j0, int nh, int c0, float (&s_m)[kWarps][kNH], float (&s_l)[kWarps][kNH]) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;  // packed row bytes
  constexpr int CPR = RB / 16;             // 16-byte chunks per packed row
  TailSmem& ts = sm.tail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = min(kTailTok, p.l - c0);
  const int nk = max(0, min(n, p.nq_k - c0));  // rows [0, nk) hold packed keys
  const int nv = max(0, min(n, p.nq_v - c0));  // rows [0, nv) hold packed values

  // ---- stage the round (c0 is a multiple of 32, so its packed keys span at
  //      most two key groups), and q ----
  for (int i = tid; i < n * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    const long t = c0 + r;
    const uint8_t* tile = tile_at<BITS>(cv, unit, t / kGroup);
    const int tr = (int)(t % kGroup);  // row within the tile
    if (r < nk) {
      if (c < CPR) cp_async16(&ts.krow[r][c], tile + tr * RB + 16 * krow_chunk<BITS>(tr, c));
    } else {
      cp_async16(&ts.krow[r][c ^ (r & 7)], cv.ring_k + (unit * cv.W + t % cv.W) * kHeadDim + 8 * c);
    }
    if (r < nv) {
      if (c < CPR) {
        cp_async16(&ts.vrow[r][c], tile + kOffVc<BITS> + tr * RB + 16 * vrow_chunk<BITS>(tr, c));
      }
    } else {
      cp_async16(&ts.vrow[r][c ^ (r & 7)], cv.ring_v + (unit * cv.W + t % cv.W) * kHeadDim + 8 * c);
    }
  }
  // key scale / zero blocks of the packed key tiles, value scale / zero
  // blocks of the packed value tiles (at most two tiles each)
  const int ngk = (nk + kGroup - 1) / kGroup, ngv = (nv + kGroup - 1) / kGroup;
  const int ocb = outlier_block_bytes(cv.n_out) / 16;  // 16-byte chunks of an outlier block
  for (int i = tid; i < ngk * ocb; i += blockDim.x) {
    const int gi = i / ocb, c = i % ocb;
    cp_async16(&ts.ko[gi][4 * c], tile_at<BITS>(cv, unit, c0 / kGroup + gi) + kTileBytes<BITS> + 16 * c);
  }
  for (int i = tid; i < (ngk + ngv) * 32; i += blockDim.x) {
    const bool key = i < ngk * 32;
    const int ii = key ? i : i - ngk * 32;
    const int gi = ii >> 5, arr = (ii >> 4) & 1, c = ii & 15;
    const uint8_t* tile = tile_at<BITS>(cv, unit, c0 / kGroup + gi);
    if (key) cp_async16(&ts.kg[gi][arr][4 * c], tile + (arr ? kOffZk<BITS> : kOffSk<BITS>) + 16 * c);
    else cp_async16(&ts.vg[gi][arr][4 * c], tile + (arr ? kOffZv<BITS> : kOffSv<BITS>) + 16 * c);
  }
  cp_async_commit();
  {
    float qj[kNH];
#pragma unroll
    for (int j = 0; j < kNH; ++j)
      qj[j] = j < nh ? load_q(a.q, ((long)b * a.Hq + j0 + j) * kHeadDim + tid, a.q_dtype) * a.scale_log2 : 0.0f;
    ts.q4[tid] = make_float4(qj[0], qj[1], qj[2], qj[3]);
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- scores: thread (token r, quarter qq) sums channels 32qq .. +31 ----
#pragma unroll 1
  for (int it = 0; it < kTailTok / 32; ++it) {
    const int r = (tid >> 2) + 32 * it, qq = tid & 3;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nk) {
      const int gi = r >> 5;
      const uint32_t* cw4 = reinterpret_cast<const uint32_t*>(&ts.krow[r][0]) + qq * BITS;
      // channels 32qq .. 32qq + 31 (kscale_pos keeps them in this block)
      const __half* sk = reinterpret_cast<const __half*>(ts.kg[gi][0]) + 32 * qq;
      const __half* zk = reinterpret_cast<const __half*>(ts.kg[gi][1]) + 32 * qq;
      if constexpr (BITS == 3) {
        // low two bits from the 2-bit plane, the high bit from its unit
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(&ts.krow[r][0]);
#pragma unroll 4
        for (int dq = 0; dq < 32; dq += 2) {
          const float2 sp = make_float2(__half2float(sk[kscale_pos<BITS>(dq)]),
                                        __half2float(sk[kscale_pos<BITS>(dq + 1)]));
          const float2 zp = make_float2(__half2float(zk[kscale_pos<BITS>(dq)]),
                                        __half2float(zk[kscale_pos<BITS>(dq + 1)]));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 32 * qq + dq + u;  // the channel
            const uint32_t lo = (kr[e >> 4] >> (2 * (e & 15))) & 3u;
            const uint32_t hi =
                (kr[kHiPlane3 / 4 + ((e >> 4) & 3)] >> (16 * ((e >> 3) & 1) + hi_bit3(e >> 6, e & 7))) & 1u;
            const float kx = fmaf((float)(lo | (hi << 2)), u ? sp.y : sp.x, u ? zp.y : zp.x);
            const float4 qv = ts.q4[e];
            acc.x = fmaf(kx, qv.x, acc.x);
            acc.y = fmaf(kx, qv.y, acc.y);
            acc.z = fmaf(kx, qv.z, acc.z);
            acc.w = fmaf(kx, qv.w, acc.w);
          }
        }
      } else {
#pragma unroll
      for (int w = 0; w < BITS; ++w) {  // 32-bit words of this quarter's codes
        const uint32_t cw = cw4[w];
#pragma unroll
        for (int e = 0; e < 32 / BITS; e += 2) {
          const int dq = w * (32 / BITS) + e;  // even channel of the quarter
          const float2 sp = make_float2(__half2float(sk[kscale_pos<BITS>(dq)]),
                                        __half2float(sk[kscale_pos<BITS>(dq + 1)]));
          const float2 zp = make_float2(__half2float(zk[kscale_pos<BITS>(dq)]),
                                        __half2float(zk[kscale_pos<BITS>(dq + 1)]));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            // the code as an exact float: its bits under the exponent of 2^23
            const float cf = __uint_as_float(((cw >> (BITS * (e + u))) & L) | 0x4B000000u) - 8388608.0f;
            const float kx = fmaf(cf, u ? sp.y : sp.x, u ? zp.y : zp.x);
            const float4 qv = ts.q4[32 * qq + dq + u];
            acc.x = fmaf(kx, qv.x, acc.x);
            acc.y = fmaf(kx, qv.y, acc.y);
            acc.z = fmaf(kx, qv.z, acc.z);
            acc.w = fmaf(kx, qv.w, acc.w);
          }
        }
      }
      }
    } else if (r < n) {
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int c = 4 * qq + c4;
        const uint4 kv = ts.krow[r][c ^ (r & 7)];
        const float kf[8] = {h_lo(kv.x), h_hi(kv.x), h_lo(kv.y), h_hi(kv.y),
                             h_lo(kv.z), h_hi(kv.z), h_lo(kv.w), h_hi(kv.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 qv = ts.q4[8 * c + e];
          acc.x = fmaf(kf[e], qv.x, acc.x);
          acc.y = fmaf(kf[e], qv.y, acc.y);
          acc.z = fmaf(kf[e], qv.z, acc.z);
          acc.w = fmaf(kf[e], qv.w, acc.w);
        }
      }
    }
#pragma unroll
    for (int sh = 1; sh <= 2; sh <<= 1) {
      acc.x += __shfl_xor_sync(kFull, acc.x, sh);
      acc.y += __shfl_xor_sync(kFull, acc.y, sh);
      acc.z += __shfl_xor_sync(kFull, acc.z, sh);
      acc.w += __shfl_xor_sync(kFull, acc.w, sh);
    }
    if (qq == 0 && r < nk && cv.n_out > 0) {
      // the group's fp16 outlier channels (their packed codes decode to 0)
      const uint32_t iw = ts.ko[r >> 5][0];
      const __half* ov = reinterpret_cast<const __half*>(&ts.ko[r >> 5][4]);
      for (int o = 0; o < cv.n_out; ++o) {
        const float x = __half2float(ov[(r & 31) * cv.n_out + o]);
        const float4 qv = ts.q4[(iw >> (8 * o)) & 0xffu];
        acc.x = fmaf(x, qv.x, acc.x);
        acc.y = fmaf(x, qv.y, acc.y);
        acc.z = fmaf(x, qv.z, acc.z);
        acc.w = fmaf(x, qv.w, acc.w);
      }
    }
    if (qq == 0 && r < n) ts.p4[r] = acc;
  }
  __syncthreads();

  // ---- softmax of head `warp` over the round ----
  {
    const int j = warp;  // kWarps == kNH
    float* pj = reinterpret_cast<float*>(ts.p4) + j;
    const float x0 = lane < n ? pj[4 * lane] : -INFINITY;
    const float x1 = lane + 32 < n ? pj[4 * (lane + 32)] : -INFINITY;
    const float mx = warp_max(fmaxf(x0, x1));
    const float e0 = lane < n ? fast_exp2(x0 - mx) : 0.0f;
    const float e1 = lane + 32 < n ? fast_exp2(x1 - mx) : 0.0f;
    pj[4 * lane] = e0;
    pj[4 * (lane + 32)] = e1;
    const float sum = warp_sum(e0 + e1);
    if (lane == 0) {
      ts.mh[j] = mx;
      ts.lh[j] = sum;
    }
  }
  __syncthreads();

  // ---- values: thread d accumulates channel d of the kNH heads ----
  const int d = tid;
  const int vpos = v_unit_pos(d >> 2);
  const int vsh = BITS * (d & 3);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int r = 0; r < n; ++r) {
    float vx;
    if (r < nv) {
      const uint8_t* row = reinterpret_cast<const uint8_t*>(&ts.vrow[r][0]);
      uint32_t cb;
      if constexpr (BITS == 2) cb = row[vpos];
      else if constexpr (BITS == 3) cb = row[vpos] | ((uint32_t)*reinterpret_cast<const uint16_t*>(row + kHiPlane3 + 2 * ((d & 31) >> 2)) << 8);
      else if constexpr (BITS == 4) cb = *reinterpret_cast<const uint16_t*>(row + 2 * vpos);
      else cb = *reinterpret_cast<const uint32_t*>(row + 4 * vpos);
      const int vs = vscale_pos(r & 31, d >> 5);
      const float sv = __half2float(reinterpret_cast<const __half*>(ts.vg[r >> 5][0])[vs]);
      const float zv = __half2float(reinterpret_cast<const __half*>(ts.vg[r >> 5][1])[vs]);
      float cf;
      if constexpr (BITS == 3) {
        // low two bits from the unit's byte, the high bit from bits 8.. (the high unit)
        const uint32_t lo = (cb >> (2 * (d & 3))) & 3u;
        const uint32_t hi = (cb >> (8 + hi_bit3(d >> 6, 4 * ((d >> 5) & 1) + (d & 3)))) & 1u;
        cf = (float)(lo | (hi << 2));
      } else {
        cf = __uint_as_float(((cb >> vsh) & L) | 0x4B000000u) - 8388608.0f;
      }
      vx = fmaf(cf, sv, zv);
    } else {
      const __half* row = reinterpret_cast<const __half*>(&ts.vrow[r][(d >> 3) ^ (r & 7)]);
      vx = __half2float(row[d & 7]);
    }
    const float4 pr = ts.p4[r];
    o.x = fmaf(pr.x, vx, o.x);
    o.y = fmaf(pr.y, vx, o.y);
    o.z = fmaf(pr.z, vx, o.z);
    o.w = fmaf(pr.w, vx, o.w);
  }
  __syncthreads();  // every thread is done with the staged rows (the merge area)

  float* mo0 = merge_area(sm, 0, kPathTail);
  mo0[0 * kHeadDim + d] = o.x;
  mo0[1 * kHeadDim + d] = o.y;
  mo0[2 * kHeadDim + d] = o.z;
  mo0[3 * kHeadDim + d] = o.w;
  if (lane < kNH) {
    s_m[warp][lane] = warp == 0 ? ts.mh[lane] : -INFINITY;
    s_l[warp][lane] = warp == 0 ? ts.lh[lane] : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Tensor-core path (packed tiles, 2 or 4 bits).

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Code position I (bit pair at 2 bits, nibble at 4 bits) of both 16-bit
// halves of w, kept in place: read as fp16 (exponent field zero) the pair is
// the exact subnormal pair {c_lo * base^e * 2^-24, c_hi * base^e * 2^-24}.
// Positions whose bits would reach the exponent field come from w_sh (w >> 10
// at 2 bits, w >> 8 at 4 bits).  code_exp(I) is the resulting e; the base is
// 4 at 2 bits and 16 at 4 bits.
template <int BITS, int I>
__device__ __forceinline__ uint32_t ext(uint32_t w, uint32_t w_sh) {
  if constexpr (BITS == 2) {
    static_assert(I >= 0 && I < 8, "eight bit pairs per half");
    if constexpr (I <= 4) return w & (0x00030003u << (2 * I));
    else return w_sh & (0x00030003u << (2 * (I - 5)));
  } else if constexpr (BITS == 4) {
    static_assert(I >= 0 && I < 4, "four nibbles per half");
    if constexpr (I <= 1) return w & (0x000F000Fu << (4 * I));
    else return w_sh & (0x000F000Fu << (4 * (I - 2)));
  } else {
    static_assert(I >= 0 && I < 2, "two bytes per half");
    return (I == 0 ? w : w_sh) & 0x00FF00FFu;
  }
}

// The 3-bit code at position I (0..7) of a 2-bit word's halves: its low two
// bits from lo (I < 4) or lo >> 8 (I >= 4), its high bit from hi (I < 4) or
// hi >> 1 (I >= 4), where hi is the word's high-plane unit arranged so that
// the high bit sits just above the low bits (see hi_bit3).  Read as fp16 the
// pair is {c_lo * 4^e * 2^-24, c_hi * 4^e * 2^-24}, e = I mod 4.
template <int I>
__device__ __forceinline__ uint32_t ext3(uint32_t lo, uint32_t lo_sh, uint32_t hi, uint32_t hi_sh) {
  static_assert(I >= 0 && I < 8, "eight code positions per half");
  constexpr uint32_t ml = 0x00030003u << (2 * (I & 3)), mh = 0x00040004u << (2 * (I & 3));
  return ((I < 4 ? lo : lo_sh) & ml) | ((I < 4 ? hi : hi_sh) & mh);
}

// Bytes swapped within each 16-bit half (set 1 of a high-plane unit).
__device__ __forceinline__ uint32_t swap_half_bytes(uint32_t x) { return __byte_perm(x, 0u, 0x2301); }

// Byte J of a and of b as the fp16 pair {a_J * 2^-24, b_J * 2^-24} (an 8-bit
// code in the low byte of each half, exponent field zero).
template <int J>
__device__ __forceinline__ uint32_t byte_pair(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, J | (J << 4) | ((4 + J) << 8) | ((4 + J) << 12)) & 0x00FF00FFu;
}

template <int BITS>
__host__ __device__ constexpr int code_exp(int i) {
  return BITS == 2 ? (i <= 4 ? i : i - 5) : (BITS == 3 ? (i & 3) : (BITS == 4 ? (i & 1) : 0));
}

template <int BITS>
constexpr int kShift = BITS == 2 ? 10 : 8;  // w_sh = w >> kShift

// base^-e(i) as a float; the base is 2^BITS, and 4 at 3 bits (whose low
// bits sit on the 2-bit grid, the high bit just above them)
template <int BITS>
__host__ __device__ constexpr float code_scale(int i) {
  return 1.0f / (float)(1 << ((BITS == 3 ? 2 : BITS) * code_exp<BITS>(i)));
}

constexpr float kTwo24 = 16777216.0f;  // undoes the 2^-24 of the subnormal codes
// The running max of a head is raised only when a tile's scores exceed it by
// more than this (log2 units), so p <= 2^0.5 and p * s stays below the fp16
// maximum for any fp16 scale s = range / 3.
constexpr float kLazyMax = 0.5f;
// A raised running max is set this far above the tile max (log2 units), so
// that later tiles rarely raise it again.
constexpr float kLazySlack = 1.0f;

// The channel-pair words of a per-channel fp16 vector stored in pair order
// (key scales or zeros, see kscale_pos) behind q-table block `blk` of this
// lane: pair block m = tig + 4 blk, whose word i is the pair of code position
// i -- 2 bits: channels (16m + i, 16m + 8 + i), i < 8; 4 bits: (8m + i, 8m +
// 4 + i), i < 4.
//
// 8 bits: pair blocks of 4 channels, words (4m, 4m + 2) and (4m + 1, 4m + 3)
// at word 2m and 2m + 1; k-step ks of lane tig takes block m = 8 tig + ks, so
// block `blk` (k-steps 2 blk, 2 blk + 1) is the 4 words from 16 tig + 4 blk.
template <int BITS>
__device__ __forceinline__ void pair_words(const uint32_t* vec, int tig, int blk, uint32_t (&P)[8]) {
  if constexpr (BITS == 2 || BITS == 3) {
    const int m = tig + 4 * blk;
    const uint4 wa = *reinterpret_cast<const uint4*>(vec + 8 * m);
    const uint4 wb = *reinterpret_cast<const uint4*>(vec + 8 * m + 4);
    P[0] = wa.x; P[1] = wa.y; P[2] = wa.z; P[3] = wa.w;
    P[4] = wb.x; P[5] = wb.y; P[6] = wb.z; P[7] = wb.w;
  } else {
    const int m = tig + 4 * blk;
    const uint4 wa = *reinterpret_cast<const uint4*>(vec + (BITS == 4 ? 4 * m : 16 * tig + 4 * blk));
    P[0] = wa.x; P[1] = wa.y; P[2] = wa.z; P[3] = wa.w;
    P[4] = P[5] = P[6] = P[7] = 0u;
  }
}

template <int BITS>
constexpr int kBlocks = BITS <= 3 ? 2 : 4;       // q-table blocks
template <int BITS>
constexpr int kQuartersPerBlock = BITS <= 3 ? 2 : 1;

// Code position of q-table word w (0..15).
template <int BITS>
__host__ __device__ constexpr int word_pos(int w) {
  return BITS <= 3 ? (w & 7) : (w & 3);
}

// Q' = q * sK of one key group as MMA B fragments for column g of this lane
// (head g >> 1, part g & 1), in the order of the q tables.  The q table is
// pre-scaled by base^-e(i) to cancel the power that the code extraction
// leaves in the A operand.
template <int BITS>
__device__ __forceinline__ void build_qprime(const WarpSmem<BITS>& ws, const uint32_t* sk, int g, int tig,
                                             uint32_t (&bq)[8][2]) {
#pragma unroll
  for (int blk = 0; blk < kBlocks<BITS>; ++blk) {
    uint32_t P[8];
    pair_words<BITS>(sk, tig, blk, P);
#pragma unroll
    for (int qq = 0; qq < kQuartersPerBlock<BITS>; ++qq) {
      const int quarter = kQuartersPerBlock<BITS> * blk + qq;
      const uint4 x0 = ws.qs[0][quarter][g][tig];
      const uint4 x1 = ws.qs[1][quarter][g][tig];
      const uint32_t X0[4] = {x0.x, x0.y, x0.z, x0.w}, X1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int wq = 0; wq < 4; ++wq) {
        const int w = 4 * quarter + wq;  // table word: k-step w >> 1, half w & 1
        bq[w >> 1][w & 1] =
            split_mul(X0[wq], X1[wq], P[word_pos<BITS>(w)]);
      }
    }
  }
}

// Position of token t (0..31) in a warp's weight buffer: the value product
// reads tokens t0 = 16kk + 8aa + tig and t0 + 4 as one 8-byte pair.
__device__ __forceinline__ int pbuf_pos(int t) {
  return 8 * (t & 3) + 4 * (t >> 4) + 2 * ((t >> 3) & 1) + ((t >> 2) & 1);
}

// Scores of one staged 32-token tile for the four heads of the CTA: lane
// (g, tig) gets head tig at tokens g + 8r (sc[r], log2 units);
// ks = 2^E_tig * scale * log2(e).
template <int BITS>
__device__ __forceinline__ void key_scores(const WarpSmem<BITS>& ws, const TileBuf<BITS>& tb, int g, int tig,
                                           float ks, int n_out, float scale_log2, float (&sc)[4]) {
  constexpr int RW = 4 * BITS;  // 32-bit words per code row
  // ---- beta = zK x q: every A row is the zero vector, so D[., (tig, part)] = beta ----
  float beta4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int blk = 0; blk < kBlocks<BITS>; ++blk) {
    uint32_t P[8];
    pair_words<BITS>(tb.zk, tig, blk, P);
#pragma unroll
    for (int qq = 0; qq < kQuartersPerBlock<BITS>; ++qq) {
      const int quarter = kQuartersPerBlock<BITS> * blk + qq;
      const uint4 qb = ws.qb[quarter][g][tig];
      const uint32_t QB[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {  // the quarter's two k-steps
        const int w0 = 4 * quarter + 2 * kh;
        const uint32_t z0 = P[word_pos<BITS>(w0)];
        const uint32_t z1 = P[word_pos<BITS>(w0 + 1)];
        mma16816(beta4, z0, z0, z1, z1, QB[2 * kh], QB[2 * kh + 1]);
      }
    }
  }
  const float kb = (beta4[0] + beta4[1]) * ks;
  const float k24 = ks * kTwo24;

  // ---- scores S = codes x Q' + beta ----
  uint32_t bq[8][2];
  build_qprime<BITS>(ws, tb.sk, g, tig, bq);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint32_t* rg = tb.kc + (16 * mt + g) * RW;      // key row 16mt + g
    const uint32_t* r8 = tb.kc + (16 * mt + g + 8) * RW;  // key row 16mt + g + 8
    // words of a row this lane reads: tig + 4j at 2 and 4 bits; at 8 bits the
    // 8 words from 8 tig, as two 16-byte chunks of the (rotated) row
    constexpr int NW = BITS == 3 ? 2 : BITS;
    uint32_t wg[NW], w8[NW], sg[NW], s8[NW];
    if constexpr (BITS == 3) {
      // low planes: words tig, tig + 4 (as at 2 bits); high plane: word tig,
      // unit 2 tig + half, holding the high bits of both words
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        wg[j] = rg[tig + 4 * j];
        w8[j] = r8[tig + 4 * j];
      }
    } else if constexpr (BITS == 8) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 a0 = reinterpret_cast<const uint4*>(rg)[krow_chunk<8>(g, 2 * tig + h)];
        const uint4 a1 = reinterpret_cast<const uint4*>(r8)[krow_chunk<8>(g + 8, 2 * tig + h)];
        wg[4 * h] = a0.x; wg[4 * h + 1] = a0.y; wg[4 * h + 2] = a0.z; wg[4 * h + 3] = a0.w;
        w8[4 * h] = a1.x; w8[4 * h + 1] = a1.y; w8[4 * h + 2] = a1.z; w8[4 * h + 3] = a1.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NW; ++j) {
        wg[j] = rg[tig + 4 * j];
        w8[j] = r8[tig + 4 * j];
      }
    }
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      sg[j] = wg[j] >> kShift<BITS>;
      s8[j] = w8[j] >> kShift<BITS>;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (BITS == 3) {
      const uint32_t hg0 = rg[kHiPlane3 / 4 + tig], h80 = r8[kHiPlane3 / 4 + tig];
      const uint32_t hg1 = swap_half_bytes(hg0), h81 = swap_half_bytes(h80);
      // high sources of word j (set j): h, h >> 1
      const uint32_t hg[2] = {hg0, hg1}, h8[2] = {h80, h81};
      const uint32_t hgs[2] = {hg0 >> 1, hg1 >> 1}, h8s[2] = {h80 >> 1, h81 >> 1};
#define KIVI_KSTEP3(KS, I)                                                                                  \
  mma16816(acc, ext3<I>(wg[(KS) >> 2], sg[(KS) >> 2], hg[(KS) >> 2], hgs[(KS) >> 2]),                     \
           ext3<I>(w8[(KS) >> 2], s8[(KS) >> 2], h8[(KS) >> 2], h8s[(KS) >> 2]),                          \
           ext3<I + 1>(wg[(KS) >> 2], sg[(KS) >> 2], hg[(KS) >> 2], hgs[(KS) >> 2]),                      \
           ext3<I + 1>(w8[(KS) >> 2], s8[(KS) >> 2], h8[(KS) >> 2], h8s[(KS) >> 2]), bq[KS][0], bq[KS][1]);
      KIVI_KSTEP3(0, 0) KIVI_KSTEP3(1, 2) KIVI_KSTEP3(2, 4) KIVI_KSTEP3(3, 6)
      KIVI_KSTEP3(4, 0) KIVI_KSTEP3(5, 2) KIVI_KSTEP3(6, 4) KIVI_KSTEP3(7, 6)
#undef KIVI_KSTEP3
    } else if constexpr (BITS == 2) {
#define KIVI_KSTEP(KS, I)                                                                       \
  mma16816(acc, ext<2, I>(wg[(KS) >> 2], sg[(KS) >> 2]), ext<2, I>(w8[(KS) >> 2], s8[(KS) >> 2]), \
           ext<2, I + 1>(wg[(KS) >> 2], sg[(KS) >> 2]), ext<2, I + 1>(w8[(KS) >> 2], s8[(KS) >> 2]), \
           bq[KS][0], bq[KS][1]);
      KIVI_KSTEP(0, 0) KIVI_KSTEP(1, 2) KIVI_KSTEP(2, 4) KIVI_KSTEP(3, 6)
      KIVI_KSTEP(4, 0) KIVI_KSTEP(5, 2) KIVI_KSTEP(6, 4) KIVI_KSTEP(7, 6)
#undef KIVI_KSTEP
    } else if constexpr (BITS == 4) {
#define KIVI_KSTEP(KS, I)                                                                       \
  mma16816(acc, ext<4, I>(wg[(KS) >> 1], sg[(KS) >> 1]), ext<4, I>(w8[(KS) >> 1], s8[(KS) >> 1]), \
           ext<4, I + 1>(wg[(KS) >> 1], sg[(KS) >> 1]), ext<4, I + 1>(w8[(KS) >> 1], s8[(KS) >> 1]), \
           bq[KS][0], bq[KS][1]);
      KIVI_KSTEP(0, 0) KIVI_KSTEP(1, 2) KIVI_KSTEP(2, 0) KIVI_KSTEP(3, 2)
      KIVI_KSTEP(4, 0) KIVI_KSTEP(5, 2) KIVI_KSTEP(6, 0) KIVI_KSTEP(7, 2)
#undef KIVI_KSTEP
    } else {
      // k-step ks: word ks (channels 4m .. 4m + 3, m = 8 tig + ks), bytes 0 / 2
      // then bytes 1 / 3 of each half
#pragma unroll
      for (int ksi = 0; ksi < 8; ++ksi)
        mma16816(acc, ext<8, 0>(wg[ksi], sg[ksi]), ext<8, 0>(w8[ksi], s8[ksi]), ext<8, 1>(wg[ksi], sg[ksi]),
                 ext<8, 1>(w8[ksi], s8[ksi]), bq[ksi][0], bq[ksi][1]);
    }
    sc[2 * mt] = fmaf(acc[0] + acc[1], k24, kb);      // token 16mt + g
    sc[2 * mt + 1] = fmaf(acc[2] + acc[3], k24, kb);  // token 16mt + g + 8
  }
  if (n_out > 0) {
    // fp16 outlier channels (their codes, scales and zeros are 0 above)
    const uint32_t iw = tb.outl[0];
    const __half* ov = reinterpret_cast<const __half*>(&tb.outl[4]);  // [32 tokens][n_out]
#pragma unroll
    for (int o = 0; o < kMaxOutliers; ++o)
      if (o < n_out) {
        const float qo = ws.qv[tig][(iw >> (8 * o)) & 0xffu] * scale_log2;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int t = 16 * (r >> 1) + g + 8 * (r & 1);
          sc[r] = fmaf(qo, __half2float(ov[t * n_out + o]), sc[r]);
        }
      }
  }
}

// Online softmax of head tig over one tile's scores (8 lanes share a head):
// when a score exceeds the running max by more than kLazyMax, the max is
// raised to the tile max plus kLazySlack and what the earlier tiles left in
// lsum, O and Z is rescaled.  The weights p = 2^(S - max) <= 2^kLazyMax go to
// the warp's weight buffer.
__device__ __forceinline__ void softmax_p(const float (&sc)[4], float* pb, int g, int tig, float& m_run,
                                          float& lsum, float (&O)[8][4], float (&Z)[4]) {
  float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
  if (__any_sync(kFull, tmax > m_run + kLazyMax)) {
    const float mnew = tmax > m_run + kLazyMax ? tmax + kLazySlack : m_run;
    const float corr = fast_exp2(m_run - mnew);  // 0 on the first tile
    m_run = mnew;
    lsum *= corr;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) O[mt][i] *= corr;
#pragma unroll
    for (int i = 0; i < 4; ++i) Z[i] *= corr;
  }
  float* prow = pb + tig * 34;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float p = fast_exp2(sc[r] - m_run);  // token g + 8r
    lsum += p;
    prow[pbuf_pos(g + 8 * r)] = p;
  }
}

// Values of one staged tile: O += codes^T x (p * sV), Z += zV^T x p, with p
// from the warp's weight buffer (O and Z of head tig).  The k rows (2tig,
// 2tig+1) of k-step kk hold tokens t0 = 16kk + tig and t0 + 4, rows (2tig+8,
// 2tig+9) tokens t0 + 8 and t0 + 12.  M-tile 2gp + hm covers value group gp:
// row g is channel 32gp + 4g + 2hm, row g + 8 the next channel.
template <int BITS>
__device__ __forceinline__ void value_acc(const TileBuf<BITS>& tb, const float* pb, int g, int tig,
                                          float (&O)[8][4], float (&Z)[4]) {
  constexpr int RW = 4 * BITS;  // 32-bit words per code row
  const int part = g & 1;
  const float* pv = pb + (g >> 1) * 34 + 8 * tig;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    // u[aa][gp]: the codes of channels 4g..4g+3 of group gp for tokens (t0,
    // t0 + 4), as the two 16-bit halves (2 bits: a byte per group, two groups
    // per word)
    uint32_t pa[2], Pp[4][2], az[2], u[2][4];
    uint32_t v8a[2][4], v8b[2][4];  // 8 bits: unit words of groups 0..3 of tokens t0 and t0 + 4
    uint32_t hv[2][2];              // 3 bits: high units of tokens (t0, t0 + 4), groups 0/1 and 2/3
#pragma unroll
    for (int aa = 0; aa < 2; ++aa) {
      const int t0 = 16 * kk + 8 * aa + tig;  // tokens t0, t0 + 4
      const float2 x = *reinterpret_cast<const float2*>(pv + 4 * kk + 2 * aa);
      const uint32_t h = f2_to_h2(x.x, x.y);
      const uint32_t l = f2_to_h2(x.x - h_lo(h), x.y - h_hi(h));
      // split_mul operands of this lane's part (see split_mul)
      pa[aa] = part ? l : h;
      const uint32_t pbh = part ? h : 0u;
      // the scale / zero words of token pair (t0, t0 + 4) (see vscale_pos)
      const int pw = 4 * (4 * (2 * kk + aa) + tig);
      const uint4 S = *reinterpret_cast<const uint4*>(tb.sv + pw);  // groups 0..3
      Pp[0][aa] = split_mul(pa[aa], pbh, S.x);
      Pp[1][aa] = split_mul(pa[aa], pbh, S.y);
      Pp[2][aa] = split_mul(pa[aa], pbh, S.z);
      Pp[3][aa] = split_mul(pa[aa], pbh, S.w);
      az[aa] = tb.zv[pw + (g & 3)];
      if constexpr (BITS == 2 || BITS == 3) {
        // interleaved word g of a row holds, per byte, channels 4g..4g+3 of groups 0..3
        const uint32_t w0 = tb.vc[t0 * RW + g], w1 = tb.vc[(t0 + 4) * RW + g];
        u[aa][0] = __byte_perm(w0, w1, 0x5410);  // groups 0, 1
        u[aa][1] = __byte_perm(w0, w1, 0x7632);  // groups 2, 3
        u[aa][2] = u[aa][3] = 0u;
        if constexpr (BITS == 3) {
          // high unit g (channels 4g..4g+3 of the four groups) of both tokens;
          // groups 2, 3 (set 1) with the bytes of each half swapped
          const uint32_t a0 = tb.vc[t0 * RW + kHiPlane3 / 4 + (g >> 1)];
          const uint32_t a1 = tb.vc[(t0 + 4) * RW + kHiPlane3 / 4 + (g >> 1)];
          hv[aa][0] = __byte_perm(a0, a1, (g & 1) ? 0x7632 : 0x5410);
          hv[aa][1] = swap_half_bytes(hv[aa][0]);
        }
      } else if constexpr (BITS == 8) {
        // interleaved words 4g .. 4g + 3 of a row (logical chunk g of the
        // rotated row) hold channels 4g..4g+3 of groups 0..3, a byte each
        const uint4 w0 = reinterpret_cast<const uint4*>(tb.vc + t0 * RW)[vrow_chunk<8>(t0, g)];
        const uint4 w1 = reinterpret_cast<const uint4*>(tb.vc + (t0 + 4) * RW)[vrow_chunk<8>(t0 + 4, g)];
        v8a[aa][0] = w0.x; v8a[aa][1] = w0.y; v8a[aa][2] = w0.z; v8a[aa][3] = w0.w;
        v8b[aa][0] = w1.x; v8b[aa][1] = w1.y; v8b[aa][2] = w1.z; v8b[aa][3] = w1.w;
      } else {
        // interleaved words 2g, 2g+1 of a row hold, per 16-bit half,
        // channels 4g..4g+3 of groups 0..3
        const uint2 w0 = *reinterpret_cast<const uint2*>(tb.vc + t0 * RW + 2 * g);
        const uint2 w1 = *reinterpret_cast<const uint2*>(tb.vc + (t0 + 4) * RW + 2 * g);
        u[aa][0] = __byte_perm(w0.x, w1.x, 0x5410);
        u[aa][1] = __byte_perm(w0.x, w1.x, 0x7632);
        u[aa][2] = __byte_perm(w0.y, w1.y, 0x5410);
        u[aa][3] = __byte_perm(w0.y, w1.y, 0x7632);
      }
    }
    // z-term: rows = value groups (g & 3), columns = (head, part) of p
    mma16816(Z, az[0], az[0], az[1], az[1], pa[0], pa[1]);
    if constexpr (BITS == 3) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t x0 = u[0][half], x1 = u[1][half];
        const uint32_t x0s = x0 >> 8, x1s = x1 >> 8;
        const uint32_t h0 = hv[0][half], h1 = hv[1][half];
        const uint32_t h0s = h0 >> 1, h1s = h1 >> 1;
        // m-tiles 4*half + {0,1,2,3}: groups 2*half (positions 0..3) and 2*half+1 (4..7)
#define KIVI_VTILE3(MT, I, GP)                                                                       \
  mma16816(O[MT], ext3<I>(x0, x0s, h0, h0s), ext3<I + 1>(x0, x0s, h0, h0s), ext3<I>(x1, x1s, h1, h1s), \
           ext3<I + 1>(x1, x1s, h1, h1s), Pp[GP][0], Pp[GP][1]);
        if (half == 0) {
          KIVI_VTILE3(0, 0, 0) KIVI_VTILE3(1, 2, 0) KIVI_VTILE3(2, 4, 1) KIVI_VTILE3(3, 6, 1)
        } else {
          KIVI_VTILE3(4, 0, 2) KIVI_VTILE3(5, 2, 2) KIVI_VTILE3(6, 4, 3) KIVI_VTILE3(7, 6, 3)
        }
#undef KIVI_VTILE3
      }
    } else if constexpr (BITS == 2) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t x0 = u[0][half], x1 = u[1][half];
        const uint32_t x0s = x0 >> 10, x1s = x1 >> 10;
        // m-tiles 4*half + {0,1,2,3}: groups 2*half (bit pairs 0..3) and 2*half+1 (4..7)
#define KIVI_VTILE(MT, I, GP)                                                                     \
  mma16816(O[MT], ext<2, I>(x0, x0s), ext<2, I + 1>(x0, x0s), ext<2, I>(x1, x1s),                 \
           ext<2, I + 1>(x1, x1s), Pp[GP][0], Pp[GP][1]);
        if (half == 0) {
          KIVI_VTILE(0, 0, 0) KIVI_VTILE(1, 2, 0) KIVI_VTILE(2, 4, 1) KIVI_VTILE(3, 6, 1)
        } else {
          KIVI_VTILE(4, 0, 2) KIVI_VTILE(5, 2, 2) KIVI_VTILE(6, 4, 3) KIVI_VTILE(7, 6, 3)
        }
#undef KIVI_VTILE
      }
    } else if constexpr (BITS == 8) {
      // m-tile 2gp + hm: rows g / g + 8 are byte 2hm / 2hm + 1 of the unit
      // words, k is the token pair (t0, t0 + 4) of aa = 0, then of aa = 1
#pragma unroll
      for (int gp = 0; gp < 4; ++gp) {
        mma16816(O[2 * gp], byte_pair<0>(v8a[0][gp], v8b[0][gp]), byte_pair<1>(v8a[0][gp], v8b[0][gp]),
                 byte_pair<0>(v8a[1][gp], v8b[1][gp]), byte_pair<1>(v8a[1][gp], v8b[1][gp]), Pp[gp][0], Pp[gp][1]);
        mma16816(O[2 * gp + 1], byte_pair<2>(v8a[0][gp], v8b[0][gp]), byte_pair<3>(v8a[0][gp], v8b[0][gp]),
                 byte_pair<2>(v8a[1][gp], v8b[1][gp]), byte_pair<3>(v8a[1][gp], v8b[1][gp]), Pp[gp][0],
                 Pp[gp][1]);
      }
    } else {
#pragma unroll
      for (int gp = 0; gp < 4; ++gp) {
        const uint32_t x0 = u[0][gp], x1 = u[1][gp];
        const uint32_t x0s = x0 >> 8, x1s = x1 >> 8;
        mma16816(O[2 * gp], ext<4, 0>(x0, x0s), ext<4, 1>(x0, x0s), ext<4, 0>(x1, x1s), ext<4, 1>(x1, x1s),
                 Pp[gp][0], Pp[gp][1]);
        mma16816(O[2 * gp + 1], ext<4, 2>(x0, x0s), ext<4, 3>(x0, x0s), ext<4, 2>(x1, x1s),
                 ext<4, 3>(x1, x1s), Pp[gp][0], Pp[gp][1]);
      }
    }
  }
}

// q of the CTA's heads: staged once in shared memory, per-head exponents
// (warp w takes head w), then the tables in fragment order.  Thread (head,
// tig, word) builds the pair words of both parts.
static_assert(kWarps == kNH, "warp w loads and scales head w");

// Channels 4 lane .. 4 lane + 3 of the CTA's head `warp` (zeros past the last
// head).  Issued before the first tile copies, so that the load does not
// queue behind them.
__device__ __forceinline__ void load_q4(const AttnArgs& a, int b, int j0, int nh, float (&v)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    v[i] = warp < nh ? load_q(a.q, ((long)b * a.Hq + j0 + warp) * kHeadDim + 4 * lane + i, a.q_dtype) : 0.0f;
}

template <int BITS>
__device__ void build_q_tables(WarpSmem<BITS>& s, const AttnArgs& a, const float (&v)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    *reinterpret_cast<float4*>(&s.qv[warp][4 * lane]) = make_float4(v[0], v[1], v[2], v[3]);
    const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    if (lane == 0) {
      const int be = (int)((__float_as_uint(amax) >> 23) & 0xffu);
      // amax in [2^(be-127), 2^(be-126)) for normal amax; a subnormal amax is
      // below 2^-126, a zero row keeps E = 0
      const int E = amax == 0.0f ? 0 : (be == 0 ? -126 : be - 126);
      s.qexp[warp] = E;
      s.qscale[warp] = ldexpf(a.scale_log2, E);
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kNH * 4 * 16; idx += blockDim.x) {
    const int word = idx & 15;                // ks * 2 + r
    const int tig = (idx >> 4) & 3;
    const int hh = idx >> 6;
    const int ks = word >> 1, r = word & 1;
    int c0, c1, i;  // the channel pair of the word and its code position
    if constexpr (BITS == 2 || BITS == 3) {
      const int m = tig + 4 * (ks >> 2);
      i = 2 * (ks & 3) + r;
      c0 = 16 * m + i;
      c1 = c0 + 8;
    } else if constexpr (BITS == 4) {
      const int m = tig + 4 * (ks >> 1);
      i = 2 * (ks & 1) + r;
      c0 = 8 * m + i;
      c1 = c0 + 4;
    } else {
      const int m = 8 * tig + ks;
      i = r;
      c0 = 4 * m + r;
      c1 = c0 + 2;
    }
    const float f = code_scale<BITS>(i);
    const float q0 = ldexpf(s.qv[hh][c0], -s.qexp[hh]), q1 = ldexpf(s.qv[hh][c1], -s.qexp[hh]);
    const uint32_t qh = f2_to_h2(q0, q1);
    const uint32_t ql = f2_to_h2(q0 - h_lo(qh), q1 - h_hi(qh));
    const uint32_t sh = f2_to_h2(q0 * f, q1 * f);
    const uint32_t sl = f2_to_h2(q0 * f - h_lo(sh), q1 * f - h_hi(sh));
    const int quarter = word >> 2, wq = word & 3;
    // hi lane: (xa, xb) = (hi, 0); lo lane: (lo, hi)
    reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh][tig])[wq] = sh;
    reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh][tig])[wq] = 0u;
    reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh + 1][tig])[wq] = sl;
    reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh + 1][tig])[wq] = sh;
    reinterpret_cast<uint32_t*>(&s.qb[quarter][2 * hh][tig])[wq] = qh;
    reinterpret_cast<uint32_t*>(&s.qb[quarter][2 * hh + 1][tig])[wq] = ql;
  }
}

// The stage buffer mirrors the packed tile byte for byte.
static_assert(offsetof(TileBuf<2>, outl) == kTileBytes<2> && offsetof(TileBuf<4>, outl) == kTileBytes<4> &&
                  offsetof(TileBuf<8>, outl) == kTileBytes<8>, "stage = tile (+ the largest outlier block)");
static_assert(offsetof(TileBuf<8>, vc) == kOffVc<8> && offsetof(TileBuf<8>, sk) == kOffSk<8> &&
              offsetof(TileBuf<8>, zv) == kOffZv<8>, "stage layout (8 bits)");
static_assert(offsetof(TileBuf<2>, vc) == kOffVc<2> && offsetof(TileBuf<2>, sk) == kOffSk<2> &&
              offsetof(TileBuf<2>, zk) == kOffZk<2> && offsetof(TileBuf<2>, sv) == kOffSv<2> &&
              offsetof(TileBuf<2>, zv) == kOffZv<2>, "stage layout (2 bits)");
static_assert(offsetof(TileBuf<3>, vc) == kOffVc<3> && offsetof(TileBuf<3>, sk) == kOffSk<3> &&
              offsetof(TileBuf<3>, zk) == kOffZk<3> && offsetof(TileBuf<3>, sv) == kOffSv<3> &&
              offsetof(TileBuf<3>, zv) == kOffZv<3> && offsetof(TileBuf<3>, outl) == kTileBytes<3>,
              "stage layout (3 bits)");
static_assert(offsetof(TileBuf<4>, vc) == kOffVc<4> && offsetof(TileBuf<4>, sk) == kOffSk<4> &&
              offsetof(TileBuf<4>, zk) == kOffZk<4> && offsetof(TileBuf<4>, sv) == kOffSv<4> &&
              offsetof(TileBuf<4>, zv) == kOffZv<4>, "stage layout (4 bits)");

// Copy source of one (batch, kv-head) unit: its first packed tile.
struct UnitSrc {
  const uint8_t* tiles;
  uint32_t tile_bytes;
};

template <int BITS>
__device__ __forceinline__ UnitSrc unit_src(const CacheView& cv, long unit) {
  return UnitSrc{tile_at<BITS>(cv, unit, 0), (uint32_t)cv.tile_bytes};
}

// One bulk copy of packed tile `tile` into a stage (one lane).
template <int BITS>
__device__ __forceinline__ void issue_tile(TileBuf<BITS>& tb, unsigned long long* bar, const UnitSrc& u,
                                           int tile) {
  mbar_expect_tx(bar, u.tile_bytes);
  bulk_g2s(&tb, u.tiles + (long)tile * u.tile_bytes, u.tile_bytes, bar);
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Packed tiles [tile0, tile1) of one (batch, kv-head, head chunk) on the
// tensor cores.  Warp w takes tiles tile0 + w, + kWarps, ... through its own
// ring of staged tiles (lane 0 issues the copies; no CTA barrier in the
// loop).  Leaves each warp's (max, sum) in s_m / s_l and its output in its
// merge area.
template <int BITS>
__device__ void packed_split(const CacheView& cv, const AttnArgs& a, SplitSmem<BITS>& sm, long unit, int b,
                             int j0, int nh, int tile0, int tile1, float (&s_m)[kWarps][kNH],
                             float (&s_l)[kWarps][kNH]) {
  constexpr int kStages = kStagesOf<BITS>;
  WarpSmem<BITS>& ws = sm.ws;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int n_mine = tile0 + warp < tile1 ? (tile1 - tile0 - warp + kWarps - 1) / kWarps : 0;
  TileBuf<BITS>* st = ws.st[warp];
  unsigned long long* bars = ws.bar[warp];
  float qv4[4];
  load_q4(a, b, j0, nh, qv4);

  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kStages; ++k) mbar_init(&bars[k], 1);
    mbar_fence_init();
  }
  __syncwarp();
  const UnitSrc us = unit_src<BITS>(cv, unit);
  const int t_first = tile0 + warp;  // this warp's tiles: t_first + kWarps * k
  int issued = min(n_mine, kStages);
  // the first tile before the q tables, the other stages after them: at
  // launch every warp of the GPU issues at once, and the first tile (and the
  // tables) should not queue behind the later stages.  A dependent launch
  // whose packed tiles the append may write builds the tables while the
  // append runs and issues every copy after it.
  const bool wait_first = a.pdl == kPdlAll;
  if (!wait_first && lane == 0 && issued > 0) issue_tile<BITS>(st[0], &bars[0], us, t_first);
  build_q_tables<BITS>(ws, a, qv4);
  __syncthreads();
  if (wait_first) grid_dependency_wait();
  if (lane == 0)
    for (int k = wait_first ? 0 : 1; k < issued; ++k) issue_tile<BITS>(st[k], &bars[k], us, t_first + kWarps * k);
  const float ks = ws.qscale[tig];
  float* pb = &ws.pbuf[warp][0][0];

  float O[8][4], Z[4], m_run = -INFINITY, lsum = 0.0f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) O[mt][i] = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) Z[i] = 0.0f;

  // Tile k's scores are computed one iteration ahead of its values: the
  // scores of tile k + 1 and the values of tile k form one straight-line
  // block (the wait for tile k + 1 comes first), so that their independent
  // MMA chains can interleave.  The ring is walked kStages tiles per round so
  // that every stage address is a constant.
  int done = 0;
  bool failed = false;
  float sc[4];
  if (n_mine > 0) {
    bool ok = mbar_try_wait(&bars[0], 0u);
    if (!ok) ok = mbar_wait(&bars[0], 0u);
    if (__any_sync(kFull, !ok)) {
      failed = true;
    } else {
      key_scores<BITS>(ws, st[0], g, tig, ks, cv.n_out, a.scale_log2, sc);
      softmax_p(sc, pb, g, tig, m_run, lsum, O, Z);
      __syncwarp();
    }
  }
  int k = 0;  // tile whose values are next
  while (k + 1 < n_mine && !failed) {
#pragma unroll
    for (int sg = 0; sg < kStages; ++sg) {
      // tile k sits in stage sg (k is a multiple of kStages at sg == 0)
      if (k + 1 < n_mine && !failed) {
        const int sn = sg + 1 == kStages ? 0 : sg + 1;  // stage of tile k + 1
        const uint32_t parn = (uint32_t)(((k + 1) / kStages) & 1);
        bool ok = mbar_try_wait(&bars[sn], parn);
        if (!ok) ok = mbar_wait(&bars[sn], parn);
        if (__any_sync(kFull, !ok)) {
          failed = true;
        } else {
          float scn[4];
          key_scores<BITS>(ws, st[sn], g, tig, ks, cv.n_out, a.scale_log2, scn);
          value_acc<BITS>(st[sg], pb, g, tig, O, Z);
          done = k + 1;
          __syncwarp();  // every lane is done with stage sg and the weight buffer
          if (k + kStages < n_mine) {
            if (lane == 0) {
              fence_proxy_async();
              issue_tile<BITS>(st[sg], &bars[sg], us, t_first + kWarps * (k + kStages));
            }
            ++issued;
          }
          softmax_p(scn, pb, g, tig, m_run, lsum, O, Z);
          __syncwarp();
          ++k;
        }
      }
    }
  }
  if (!failed && n_mine > 0) {
    // the last tile's values (its stage: (n_mine - 1) % kStages)
    const int sl = (n_mine - 1) % kStages;
#pragma unroll
    for (int sg = 0; sg < kStages; ++sg)
      if (sg == sl) value_acc<BITS>(st[sg], pb, g, tig, O, Z);
    done = n_mine;
  }
  if (done < n_mine) {
    // A wait timed out: record it, and let every copy still in flight land
    // before the warp's buffers are reused (each wait bounded again).
    if (lane == 0) atomicOr(a.status, 1);
    for (int kk = done; kk < issued; ++kk) mbar_wait(&bars[kk % kStages], (uint32_t)((kk / kStages) & 1));
    __syncwarp();
  }

  // ---- this warp's partial: max, sum and output of head tig ----
  // lsum of head tig over tokens g + 8r: sum over g
  lsum += __shfl_xor_sync(kFull, lsum, 4);
  lsum += __shfl_xor_sync(kFull, lsum, 8);
  lsum += __shfl_xor_sync(kFull, lsum, 16);
  if (g == 0) {
    s_m[warp][tig] = m_run;
    s_l[warp][tig] = lsum;
  }
  // z-term of value group gp for head tig sits in lane (gp, tig)
  const float zmine = Z[0] + Z[1];
  float zt[4];
#pragma unroll
  for (int gp = 0; gp < 4; ++gp) zt[gp] = __shfl_sync(kFull, zmine, 4 * gp + tig);
  float* orow = merge_area(sm, warp, kPathMma) + tig * kHeadDim;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int gp = mt >> 1, hm = mt & 1;
    // code positions of rows g and g + 8 of m-tile mt
    const int i_lo = BITS <= 3 ? 4 * (gp & 1) + 2 * hm : 2 * hm;
    const int ch = 32 * gp + 4 * g + 2 * hm;
    const float f_lo = kTwo24 * code_scale<BITS>(i_lo);
    const float f_hi = kTwo24 * code_scale<BITS>(i_lo + 1);
    orow[ch] = (O[mt][0] + O[mt][1]) * f_lo + zt[gp];
    orow[ch + 1] = (O[mt][2] + O[mt][3]) * f_hi + zt[gp];
  }
}

// Merge n <= kMergeGroup partials [n][kNH][D] (outputs) and [n][kNH][2]
// (max, sum): warp w takes head w, lane l channels 4l..4l+3; every load is
// issued before the first is used.  Returns the merged (unnormalized) output
// quad, max and sum of head `warp`.
// Count a CTA in (thread 0, after a CTA barrier that follows the CTA's
// partial writes); returns the count before.  Release: the barrier orders
// every thread's writes before this atomic, so they are visible to whichever
// CTA sees the final count.  Acquire: the CTA that sees it reads the others'
// partials after the next barrier (with L2 loads).
__device__ __forceinline__ int count_in(int* counter) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

__device__ __forceinline__ void merge_partials(const float* po, const float* pml, int n, int nh, float4& o4,
                                               float& m_out, float& l_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4 v[kMergeGroup];
#pragma unroll
  for (int k = 0; k < kMergeGroup; ++k)
    v[k] = (k < n && warp < nh)
               ? __ldcg(reinterpret_cast<const float4*>(po + ((long)k * kNH + warp) * kHeadDim) + lane)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  const float2 ml = (lane < n && warp < nh)
                        ? __ldcg(reinterpret_cast<const float2*>(pml + ((long)lane * kNH + warp) * 2))
                        : make_float2(-INFINITY, 0.0f);
  const float M = warp_max(ml.x);
  const float e = ml.x == -INFINITY ? 0.0f : fast_exp2(ml.x - M);
  l_out = warp_sum(e * ml.y);
  m_out = M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMergeGroup; ++k) {
    const float ek = __shfl_sync(kFull, e, k);
    acc.x = fmaf(ek, v[k].x, acc.x);
    acc.y = fmaf(ek, v[k].y, acc.y);
    acc.z = fmaf(ek, v[k].z, acc.z);
    acc.w = fmaf(ek, v[k].w, acc.w);
  }
  o4 = acc;
}

// The tail on the last packed split (when no tail split fits the budget):
// the warps' packed partials are merged into registers, the tail rounds run
// one after another and are folded in, and the result is left as warp 0's
// slot (the other warps' slots empty) for the CTA merge.
template <int BITS>
__device__ void fused_tail(const CacheView& cv, const AttnArgs& a, const SeqPlan p, SplitSmem<BITS>& sm,
                           long unit, int b,
                           int j0, int nh, float (&s_m)[kWarps][kNH], float (&s_l)[kWarps][kNH]) {
  const int d = threadIdx.x;
  float pm[kNH], pl[kNH], po[kNH];
#pragma unroll
  for (int j = 0; j < kNH; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][j]);
    float lt = 0.0f, ot = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (s_m[w][j] == -INFINITY) continue;
        const float e = fast_exp2(s_m[w][j] - M);
        lt += e * s_l[w][j];
        ot += e * merge_area(sm, w, kPathMma)[j * kHeadDim + d];
      }
    }
    pm[j] = M;
    pl[j] = lt;
    po[j] = ot;
  }
  __syncthreads();  // the warps' slots are read; the tail may overwrite them
  for (int c0 = p.t_tail; c0 < p.l; c0 += kTailTok) {
    tail_split<BITS>(cv, a, p, sm, unit, b, j0, nh, c0, s_m, s_l);
    __syncthreads();
    const float* mo0 = merge_area(sm, 0, kPathTail);
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      const float tm = s_m[0][j];
      const float M = fmaxf(pm[j], tm);
      const float e1 = pm[j] == -INFINITY ? 0.0f : fast_exp2(pm[j] - M);
      const float e2 = tm == -INFINITY ? 0.0f : fast_exp2(tm - M);
      po[j] = po[j] * e1 + mo0[j * kHeadDim + d] * e2;
      pl[j] = pl[j] * e1 + s_l[0][j] * e2;
      pm[j] = M;
    }
    __syncthreads();  // before the next round overwrites the staged rows
  }
  float* out0 = merge_area(sm, 0, kPathMma);
#pragma unroll
  for (int j = 0; j < kNH; ++j) out0[j * kHeadDim + d] = po[j];
  if (d < kWarps * kNH) {
    const int w = d / kNH, j = d % kNH;
    s_m[w][j] = w == 0 ? pick4(pm, j) : -INFINITY;
    s_l[w][j] = w == 0 ? pick4(pl, j) : 0.0f;
  }
  __syncthreads();
}

// grid (splits, H * head_chunks, B), 128 threads.
template <int BITS>
__global__ void __launch_bounds__(128, attn_ctas_per_sm(BITS)) attn_kernel(CacheView cv, AttnArgs a, const SeqLens lens) {
  extern __shared__ __align__(16) unsigned char smem_raw[];  // sizeof(SplitSmem<BITS>)
  SplitSmem<BITS>& sm = *reinterpret_cast<SplitSmem<BITS>*>(smem_raw);
  __shared__ float s_m[kWarps][kNH], s_l[kWarps][kNH];
  __shared__ bool s_last;

  const int s = blockIdx.x;
  const int nhc = gridDim.y / cv.H;
  const int h = blockIdx.y / nhc, hc = blockIdx.y % nhc;
  const int b = blockIdx.z;
  const int grp = a.Hq / cv.H;
  const int j0 = h * grp + hc * kNH;
  const int nh = min(kNH, grp - hc * kNH);
  const long unit = (long)b * cv.H + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this sequence's plan; splits past its own count have nothing to do (and
  // are not counted by its merge)
  const SeqPlan p = lens.uniform >= 0 ? a.plan : make_plan(lens.l[b], cv.R, cv.policy, a.scfg);
  if (s >= p.splits) return;
  const int path = s < p.tail_splits ? kPathTail : kPathMma;

  if (path == kPathTail) {
    if (a.pdl) grid_dependency_wait();  // the tail reads the rings the append writes
    tail_split<BITS>(cv, a, p, sm, unit, b, j0, nh, p.t_tail + s * kTailTok, s_m, s_l);
  } else {
    // ---- tensor cores: packed tiles [sp*chunk, min(t_tail, (sp+1)*chunk)) ----
    const int sp = s - p.tail_splits;
    const int tile0 = sp * p.chunk / 32;
    const int tile1 = min(p.t_tail, (sp + 1) * p.chunk) / 32;
    packed_split<BITS>(cv, a, sm, unit, b, j0, nh, tile0, tile1, s_m, s_l);
  }
  __syncthreads();
  if (path == kPathMma && p.tail_fused && s == p.splits - 1) {
    if (a.pdl == kPdlTail) grid_dependency_wait();  // the tail reads what the append wrote
    fused_tail<BITS>(cv, a, p, sm, unit, b, j0, nh, s_m, s_l);
  }

  // ---- merge the warps of this CTA into one partial per head ----
  const int d = threadIdx.x;
  const long gid = (long)b * gridDim.y + blockIdx.y;  // (batch, kv-head, head chunk)
  for (int j = 0; j < nh; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][j]);
    float lt = 0.0f, ot = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (s_m[w][j] == -INFINITY) continue;  // an empty warp (its area is not written)
        const float e = fast_exp2(s_m[w][j] - M);
        lt += e * s_l[w][j];
        ot += e * merge_area(sm, w, path)[j * kHeadDim + d];
      }
    }
    const long pidx = (gid * a.splits + s) * kNH + j;
    a.ws_o[pidx * kHeadDim + d] = ot;
    if (d == 0) {
      a.ws_ml[pidx * 2] = M;
      a.ws_ml[pidx * 2 + 1] = lt;
    }
  }

  // ---- the last CTA of each group of kMergeGroup splits merges the group;
  //      with more than one group, the last group merges the group results ----
  const int n_grp = (p.splits + kMergeGroup - 1) / kMergeGroup;
  const int grp_i = s / kMergeGroup;
  const int g_lo = grp_i * kMergeGroup, g_n = min(kMergeGroup, p.splits - g_lo);
  __syncthreads();
  if (threadIdx.x == 0) {
    int* counter = a.counters + gid * a.merge_groups + grp_i;
    s_last = count_in(counter) == g_n - 1;
    if (s_last) *counter = 0;  // every other CTA of the group has counted in
  }
  __syncthreads();
  if (!s_last) return;
  float4 o4;
  float lsum_h, m_h;
  merge_partials(a.ws_o + (gid * a.splits + g_lo) * kNH * kHeadDim, a.ws_ml + (gid * a.splits + g_lo) * kNH * 2,
                 g_n, nh, o4, m_h, lsum_h);
  if (n_grp > 1) {
    // a group result: write it, then count the group in
    if (warp < nh) {
      const long pidx = (gid * a.merge_groups + grp_i) * kNH + warp;
      *reinterpret_cast<float4*>(a.ws_o1 + pidx * kHeadDim + 4 * lane) = o4;
      if (lane == 0) {
        a.ws_ml1[pidx * 2] = m_h;
        a.ws_ml1[pidx * 2 + 1] = lsum_h;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int* counter = a.counters2 + gid;
      s_last = count_in(counter) == n_grp - 1;
      if (s_last) *counter = 0;
    }
    __syncthreads();
    if (!s_last) return;
    merge_partials(a.ws_o1 + gid * a.merge_groups * kNH * kHeadDim, a.ws_ml1 + gid * a.merge_groups * kNH * 2,
                   n_grp, nh, o4, m_h, lsum_h);
  }
  if (warp < nh) {
    const float inv = 1.0f / lsum_h;
    const float r[4] = {o4.x * inv, o4.y * inv, o4.z * inv, o4.w * inv};
    const long oi = ((long)b * a.Hq + j0 + warp) * kHeadDim + 4 * lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (a.q_dtype == kF32) static_cast<float*>(a.out)[oi + i] = r[i];
      else if (a.q_dtype == kF16) static_cast<__half*>(a.out)[oi + i] = __float2half_rn(r[i]);
      else static_cast<__nv_bfloat16*>(a.out)[oi + i] = __float2bfloat16_rn(r[i]);
    }
  }
}

}  // namespace

// attn_ctas_per_sm(BITS) CTAs must fit an SM's 228 KB of shared memory
// (1 KB of it reserved per CTA).
static_assert(4 * (sizeof(SplitSmem<2>) + 1024 + 256) <= 228 * 1024, "2-bit CTAs per SM");
static_assert(4 * (sizeof(SplitSmem<3>) + 1024 + 256) <= 228 * 1024, "3-bit CTAs per SM");
static_assert(4 * (sizeof(SplitSmem<4>) + 1024 + 256) <= 228 * 1024, "4-bit CTAs per SM");
static_assert(2 * (sizeof(SplitSmem<8>) + 1024 + 256) <= 228 * 1024, "8-bit CTAs per SM");

template <int BITS>
cudaError_t launch_bits(const dim3& grid, const CacheView& cv, const AttnArgs& a, const SeqLens& lens,
                        cudaStream_t st) {
  // The shared-memory opt-in is a per-device function attribute; setting it
  // on every call costs a host call only.
  const cudaError_t e = cudaFuncSetAttribute(attn_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(SplitSmem<BITS>));
  if (e != cudaSuccess) return e;
  if (!a.pdl) {
    attn_kernel<BITS><<<grid, 128, sizeof(SplitSmem<BITS>), st>>>(cv, a, lens);
    return cudaGetLastError();
  }
  // a programmatic dependent of the kernel before it on the stream
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(128);
  lc.dynamicSmemBytes = sizeof(SplitSmem<BITS>);
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, attn_kernel<BITS>, cv, a, lens);
}

cudaError_t launch_wait_probe(int* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a, const SeqLens& lens, cudaStream_t st) {
  const int grp = a.Hq / cv.H;
  const int nhc = (grp + kNH - 1) / kNH;
  const dim3 grid(a.splits, cv.H * nhc, cv.B);
  switch (cv.bits) {
    case 2: return launch_bits<2>(grid, cv, a, lens, st);
    case 3: return launch_bits<3>(grid, cv, a, lens, st);
    case 4: return launch_bits<4>(grid, cv, a, lens, st);
    default: return launch_bits<8>(grid, cv, a, lens, st);
  }
}

}  // namespace kivi
