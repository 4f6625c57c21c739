// attention.cu -- decode attention over the packed KIVI cache.
//
// Decode step 2 of the chooblog KIVI review (§1.3): A = softmax(t_Q X_K^T),
// t_O = A X_V, scaled by 1/sqrt(D) as in the notebook "KIVI - 2-bit KV cache
// quantisation"; dequantization is fused into both products (review §3.2
// "System-Level": no separate dequantize pass).
//
// The context is split along the tokens (flash-decoding).  Split 0 of every
// (batch, kv-head, head chunk) takes the tail [t_tail, l) -- the tokens whose
// keys or values are still fp16 in the residual rings, plus the partial
// value group before them -- on CUDA cores.  Splits 1.. take the fully
// packed 32-token tiles [0, t_tail).  The CTA that finishes last for a
// (batch, kv-head, head chunk) merges the partial (max, sum, output) triples,
// in the same launch; nothing ever waits.
//
// Packed tiles at 2 bits run on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulation):
//   scores  S[t, j] = sum_d c_td (q_jd s_d) + beta_j, beta_j = sum_d q_jd z_d
//   output  O[d, j] = sum_t c_td (p_jt s_t,g(d)) + sum_t p_jt z_t,g(d)
// The codes c are small integers, exact in fp16.  The fp32 factors q*s and
// p*s enter as an fp16 hi/lo pair (hi = fp16(x), lo = fp16(x - hi)), which
// fill the 8 columns of the n=8 operand as (head, hi) and (head, lo): four
// query heads per MMA, and the sum hi + lo recovers x to about 2^-22.
#include <cuda_bf16.h>

#include <cstddef>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;
constexpr int kNH = 4;      // query heads per CTA (one "head chunk")
constexpr int kStages = 3;  // cp.async pipeline depth of each warp (tensor-core path)

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

__device__ __forceinline__ void halves4(uint2 u, float (&f)[4]) {
  f[0] = h_lo(u.x);
  f[1] = h_hi(u.x);
  f[2] = h_lo(u.y);
  f[3] = h_hi(u.y);
}

__device__ __forceinline__ uint32_t h2u(__half2 h) {
  return (uint32_t)__half_as_ushort(__low2half(h)) | ((uint32_t)__half_as_ushort(__high2half(h)) << 16);
}

__device__ __forceinline__ __half2 u2h(uint32_t u) {
  return __halves2half2(__ushort_as_half((unsigned short)(u & 0xffffu)),
                        __ushort_as_half((unsigned short)(u >> 16)));
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

// x * s for an fp32 x given as an fp16 pair (xa, xb) with x = xa + xb, split
// again as hi + lo across lanes: a "hi" lane passes (xa = hi(x), xb = 0) and
// gets fp16(x * s); a "lo" lane passes (xa = lo(x), xb = hi(x)) and gets
// fp16(xa * s + (xb * s - fp16(xb * s))), the residual of the hi product being
// exact in fp16.  xbn is -xb.  Three fp16x2 instructions, no select.
__device__ __forceinline__ uint32_t split_mul(uint32_t xa, uint32_t xb, uint32_t xbn, uint32_t s) {
  return hfma2u(xa, s, hfma2u(xb, s, hmul2u(xbn, s)));
}

// Value rows are group-interleaved: the byte unit of channels 32*gp + 4*w ..
// +3 sits at unit position 4*w + gp (units are bits/2 bytes).
__device__ __forceinline__ int v_unit_pos(int unit) { return 4 * (unit & 7) + (unit >> 3); }

// ---------------------------------------------------------------------------
// Shared memory.

struct V1Smem {                           // CUDA-core path (tail, and 4-bit tiles)
  float q[kNH][kHeadDim];                 // q * scale * log2(e)
  // per warp: q * sK of its key group ([kNH][128] floats), or 32 fp16
  // residual rows (256 B each, 16-byte chunks XOR-swizzled by row), or the
  // merge area at the end
  uint4 wbuf[kWarps][32 * 16];
  uint8_t vc[kWarps][32 * 64];            // staged value codes (up to 4 bits)
  __half vsz[kWarps][32][8];              // staged value scale[4], zero[4] per row
};

// One packed 32-token tile at 2 bits.  Padding keeps the lane access
// patterns of the tensor-core path free of shared-memory bank conflicts:
// value rows are 48 B apart, and the key scales / zeros of channels 64..127
// start 16 B after those of channels 0..63.
struct TileStage {
  uint32_t kc[32 * 8];                    // key codes: 32 rows x 32 B
  uint32_t vc[32 * 12];                   // value codes: 32 rows x 32 B, 48 B stride
  uint32_t sk[68], zk[68];                // 128 fp16 key scales / zeros (+ 4-word gap)
  uint32_t sv[64], zv[64];                // [32 tokens][4 groups] fp16
};

// word index of key scale / zero word w (0..63) in the padded layout
__device__ __forceinline__ int kpad(int w) { return w + ((w >> 5) << 2); }

// q tables in MMA fragment order.  Lane (g, tig) reads the 16 words of
// column g (head g >> 1, part g & 1) for its tig, as four 16-byte quarters;
// the layout [quarter][column][tig] spreads the 8 lanes of a shared-memory
// phase over distinct banks.  Word w of (column, tig) holds channels
// (16m + i, 16m + i + 8) with ks = w >> 1, m = 2*tig + (ks >> 2),
// i = 2*(ks & 3) + (w & 1).
struct MmaSmem {
  uint4 qs[3][4][8][4];                   // q * 4^-e(d) as split_mul operands (xa, xb, xbn)
  uint4 qb[4][8][4];                      // q (unscaled) hi / lo
  TileStage st[kWarps][kStages];
};

union SplitSmem {
  V1Smem v1;
  MmaSmem mma;
};

// Per-warp merge area: [kNH][kHeadDim] floats inside the warp's own buffers,
// written only after the warp has finished its tiles.
__device__ __forceinline__ float* merge_area(SplitSmem& sm, int warp, bool mma_path) {
  return mma_path ? reinterpret_cast<float*>(&sm.mma.st[warp][0])
                  : reinterpret_cast<float*>(&sm.v1.wbuf[warp][0]);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// Stage residual rows [r0, r1) of a 32-token tile (ring slots (tt0 + r) mod R)
// into a warp buffer: chunk c of row r goes to uint4 index 16r + (c ^ (r & 7)).
__device__ __forceinline__ void stage_ring_rows(const __half* ring, long unit, int R, int tt0,
                                                int r0, int r1, uint4* buf, int lane) {
  for (int i = 16 * r0 + lane; i < 16 * r1; i += 32) {
    const int r = i >> 4, c = i & 15;
    cp_async16(&buf[16 * r + (c ^ (r & 7))],
               ring + (unit * R + (tt0 + r) % R) * kHeadDim + 8 * c);
  }
  cp_async_commit();
}

// ---------------------------------------------------------------------------
// CUDA-core path: tiles of [t_begin, t_end) that may hold fp16 residual rows.
// Warp w walks 32-token tiles w, w+4, ...; in the key phase lane l owns token
// tile+l, in the value phase lane l owns channels 4l..4l+3.
template <int BITS>
__device__ void v1_tiles(const CacheView& cv, const AttnArgs& a, SplitSmem& sm, long unit,
                         int t_begin, int t_end, float (&m)[kNH], float (&lsum)[kNH],
                         float (&o)[kNH][4]) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int CPW = 32 / BITS;
  V1Smem& s = sm.v1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* wbuf = s.wbuf[warp];
  float* qk = reinterpret_cast<float*>(wbuf);
  const int tile_end = (t_end + 31) / 32;
  for (int tile = t_begin / 32 + warp; tile < tile_end; tile += kWarps) {
    const int tt0 = tile * 32;
    const int t = tt0 + lane;
    const bool valid = t >= t_begin && t < t_end;
    float sc[kNH];
    if (tt0 + 32 <= a.nq_k) {
      // packed keys: q' = q * sK[g] (to smem), beta = q . zK[g]
      const long go = (unit * (cv.Tcap / kGroup) + tile) * kHeadDim + 4 * lane;
      float skf[4], zkf[4];
      halves4(*reinterpret_cast<const uint2*>(cv.scale_k + go), skf);
      halves4(*reinterpret_cast<const uint2*>(cv.zero_k + go), zkf);
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        const float4 qv = *reinterpret_cast<const float4*>(&s.q[j][4 * lane]);
        *reinterpret_cast<float4*>(&qk[j * kHeadDim + 4 * lane]) =
            make_float4(qv.x * skf[0], qv.y * skf[1], qv.z * skf[2], qv.w * skf[3]);
        sc[j] = warp_sum(qv.x * zkf[0] + qv.y * zkf[1] + qv.z * zkf[2] + qv.w * zkf[3]);
      }
      __syncwarp();
      if (valid) {
        const uint4* row = reinterpret_cast<const uint4*>(cv.codes_k + (unit * cv.Tcap + t) * RB);
#pragma unroll
        for (int w4 = 0; w4 < RB / 16; ++w4) {
          const uint4 cw = row[w4];
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const int dbase = (w4 * 4 + wi) * CPW;
#pragma unroll
            for (int e = 0; e < CPW; e += 4) {
              const float c0 = (float)((words[wi] >> (BITS * (e + 0))) & L);
              const float c1 = (float)((words[wi] >> (BITS * (e + 1))) & L);
              const float c2 = (float)((words[wi] >> (BITS * (e + 2))) & L);
              const float c3 = (float)((words[wi] >> (BITS * (e + 3))) & L);
#pragma unroll
              for (int j = 0; j < kNH; ++j) {
                const float4 qkv = *reinterpret_cast<const float4*>(&qk[j * kHeadDim + dbase + e]);
                sc[j] += qkv.x * c0 + qkv.y * c1 + qkv.z * c2 + qkv.w * c3;
              }
            }
          }
        }
      }
    } else {
      // residual keys: stage the fp16 ring rows, then lane = token
#pragma unroll
      for (int j = 0; j < kNH; ++j) sc[j] = 0.0f;
      stage_ring_rows(cv.ring_k, unit, cv.R, tt0, max(t_begin - tt0, 0), min(32, t_end - tt0),
                      wbuf, lane);
      cp_async_wait<0>();
      __syncwarp();
      if (valid) {
#pragma unroll 4
        for (int d8 = 0; d8 < kHeadDim; d8 += 8) {
          const uint4 kv = wbuf[16 * lane + ((d8 >> 3) ^ (lane & 7))];
          const float kf[8] = {h_lo(kv.x), h_hi(kv.x), h_lo(kv.y), h_hi(kv.y),
                               h_lo(kv.z), h_hi(kv.z), h_lo(kv.w), h_hi(kv.w)};
#pragma unroll
          for (int j = 0; j < kNH; ++j) {
            const float4 q0 = *reinterpret_cast<const float4*>(&s.q[j][d8]);
            const float4 q1 = *reinterpret_cast<const float4*>(&s.q[j][d8 + 4]);
            sc[j] += q0.x * kf[0] + q0.y * kf[1] + q0.z * kf[2] + q0.w * kf[3] +
                     q1.x * kf[4] + q1.y * kf[5] + q1.z * kf[6] + q1.w * kf[7];
          }
        }
      }
    }

    // online softmax (log2 domain: q carries scale * log2 e)
    float p[kNH];
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      const float sj = valid ? sc[j] : -INFINITY;
      const float mnew = fmaxf(m[j], warp_max(sj));
      const float corr = fast_exp2(m[j] - mnew);
      p[j] = fast_exp2(sj - mnew);
      lsum[j] = lsum[j] * corr + p[j];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] *= corr;
      m[j] = mnew;
    }

    // values: stage the packed rows and the residual rows of this tile
    const int vrows = min(max(a.nq_v - tt0, 0), 32);
    const int r_lo = max(t_begin - tt0, 0);
    const int r_hi = min(32, t_end - tt0);
    __syncwarp();  // the key phase is done with wbuf
    if (max(vrows, r_lo) < r_hi) stage_ring_rows(cv.ring_v, unit, cv.R, tt0, max(vrows, r_lo), r_hi, wbuf, lane);
    {
      const uint4* gsrc = reinterpret_cast<const uint4*>(cv.codes_v + (unit * cv.Tcap + tt0) * RB);
      uint4* sdst = reinterpret_cast<uint4*>(s.vc[warp]);
      for (int i = lane; i < vrows * RB / 16; i += 32) sdst[i] = gsrc[i];
      if (lane < vrows) {
        const long so = (unit * cv.Tcap + tt0 + lane) * (kHeadDim / kGroup);
        *reinterpret_cast<uint2*>(&s.vsz[warp][lane][0]) = *reinterpret_cast<const uint2*>(cv.scale_v + so);
        *reinterpret_cast<uint2*>(&s.vsz[warp][lane][4]) = *reinterpret_cast<const uint2*>(cv.zero_v + so);
      }
    }
    cp_async_wait<0>();
    __syncwarp();
    const int vpos = v_unit_pos(lane);  // unit of channels 4*lane .. +3
    for (int r = r_lo; r < r_hi; ++r) {
      float vh[4];
      if (r < vrows) {
        uint32_t cb;
        if constexpr (BITS == 2) cb = s.vc[warp][r * RB + vpos];
        else cb = *reinterpret_cast<const uint16_t*>(&s.vc[warp][r * RB + 2 * vpos]);
        const float sv = __half2float(s.vsz[warp][r][lane >> 3]);
        const float zv = __half2float(s.vsz[warp][r][4 + (lane >> 3)]);
#pragma unroll
        for (int i = 0; i < 4; ++i) vh[i] = (float)((cb >> (BITS * i)) & L) * sv + zv;
      } else {
        const uint2* vr = reinterpret_cast<const uint2*>(&wbuf[16 * r + ((lane >> 1) ^ (r & 7))]);
        halves4(vr[lane & 1], vh);
      }
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        const float pr = __shfl_sync(kFull, p[j], r);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[j][i] += pr * vh[i];
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Tensor-core path helpers.

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The 2-bit codes at bit pair I of both 16-bit halves of w, as the exact
// fp16 pair {c_lo * 4^I, c_hi * 4^I} (I <= 4): OR the masked bits into the
// mantissa of 1024.0 (0x6400) and subtract 1024.
template <int I>
__device__ __forceinline__ uint32_t ext(uint32_t w) {
  static_assert(I >= 0 && I <= 4, "bit pair must stay inside the fp16 mantissa");
  uint32_t v, r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w), "n"(0x00030003u << (2 * I)), "n"(0x64006400u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64006400u));
  return r;
}

// Bit pair i in 0..7 of each half of w: pairs 0..4 directly, 5..7 from w >> 10
// (scaled by 4^(i-5)).  pow4_exp(i) is the resulting power of four.
template <int I>
__device__ __forceinline__ uint32_t ext8(uint32_t w, uint32_t w_sh10) {
  if constexpr (I <= 4) return ext<I>(w);
  else return ext<I - 5>(w_sh10);
}

__host__ __device__ constexpr int pow4_exp(int i) { return i <= 4 ? i : i - 5; }

// Per-lane cp.async sources and destinations of one packed tile (keys,
// values, scales, zeros: 192 chunks of 16 B, six per lane).  The sources of
// the next tile of the same warp are the current ones plus a fixed stride.
struct TileCopy {
  const char* src[6];
  uint32_t dst[6];  // shared-memory offsets inside a TileStage
};

__device__ __forceinline__ TileCopy tile_copy_plan(const CacheView& cv, long unit, int tile, int lane) {
  TileCopy tc;
  const long row0 = unit * cv.Tcap + (long)tile * 32;
  const char* kc = reinterpret_cast<const char*>(cv.codes_k + row0 * 32);
  const char* vc = reinterpret_cast<const char*>(cv.codes_v + row0 * 32);
  const long g0 = (unit * (cv.Tcap / kGroup) + tile) * kHeadDim;
  const char* sk = reinterpret_cast<const char*>(cv.scale_k + g0);
  const char* zk = reinterpret_cast<const char*>(cv.zero_k + g0);
  const char* sv = reinterpret_cast<const char*>(cv.scale_v + row0 * (kHeadDim / kGroup));
  const char* zv = reinterpret_cast<const char*>(cv.zero_v + row0 * (kHeadDim / kGroup));
  const int c = lane & 15;
  tc.src[0] = kc + 16 * lane;
  tc.src[1] = kc + 16 * (32 + lane);
  tc.src[2] = vc + 16 * lane;
  tc.src[3] = vc + 16 * (32 + lane);
  tc.src[4] = lane < 16 ? sk + 16 * c : zk + 16 * c;
  tc.src[5] = lane < 16 ? sv + 16 * c : zv + 16 * c;
  tc.dst[0] = (uint32_t)offsetof(TileStage, kc) + 16 * lane;
  tc.dst[1] = (uint32_t)offsetof(TileStage, kc) + 16 * (32 + lane);
  // value chunk 2*row + half goes to row * 48 + 16 * half bytes
  tc.dst[2] = (uint32_t)offsetof(TileStage, vc) + (lane >> 1) * 48 + 16 * (lane & 1);
  tc.dst[3] = (uint32_t)offsetof(TileStage, vc) + (16 + (lane >> 1)) * 48 + 16 * (lane & 1);
  tc.dst[4] = (uint32_t)(lane < 16 ? offsetof(TileStage, sk) : offsetof(TileStage, zk)) + 4 * kpad(4 * c);
  tc.dst[5] = (uint32_t)(lane < 16 ? offsetof(TileStage, sv) : offsetof(TileStage, zv)) + 16 * c;
  return tc;
}

// Byte strides of the six sources when a warp moves on by kWarps tiles.
__device__ __forceinline__ void tile_copy_advance(TileCopy& tc) {
  constexpr long kCodes = (long)kWarps * 32 * 32;           // 32 rows of 32 B
  constexpr long kKGroup = (long)kWarps * kHeadDim * 2;      // one group of fp16 [128]
  constexpr long kVRows = (long)kWarps * 32 * (kHeadDim / kGroup) * 2;
  tc.src[0] += kCodes;
  tc.src[1] += kCodes;
  tc.src[2] += kCodes;
  tc.src[3] += kCodes;
  tc.src[4] += kKGroup;
  tc.src[5] += kVRows;
}

__device__ __forceinline__ void issue_tile(const TileCopy& tc, TileStage& st) {
  char* base = reinterpret_cast<char*>(&st);
#pragma unroll
  for (int i = 0; i < 6; ++i) cp_async16(base + tc.dst[i], tc.src[i]);
}

// Q' = q * sK of one key group as MMA B fragments for column g of this lane
// (head g >> 1, part g & 1).  Fragment order: k-step ks uses word m = 2*tig +
// (ks >> 2) of each key row and bit pairs i = 2*(ks & 3) and i + 1; the k
// rows (2tig, 2tig+1) hold channels (16m+i, 16m+i+8) and (2tig+8, 2tig+9) hold
// (16m+i+1, 16m+i+9).  The q table is pre-scaled by 4^-e(i) to cancel the
// power of four that the code extraction leaves in the A operand.
__device__ __forceinline__ void build_qprime(const MmaSmem& s, const TileStage& st, int hh,
                                             int part, int tig, uint32_t (&bq)[8][2]) {
#pragma unroll
  for (int mh = 0; mh < 2; ++mh) {
    const int m = 2 * tig + mh;
    const uint4 wa = *reinterpret_cast<const uint4*>(&st.sk[kpad(8 * m)]);
    const uint4 wb = *reinterpret_cast<const uint4*>(&st.sk[kpad(8 * m + 4)]);
    const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w}, B[4] = {wb.x, wb.y, wb.z, wb.w};
    uint32_t X[3][8];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const uint4 x0 = s.qs[c][2 * mh][2 * hh + part][tig];
      const uint4 x1 = s.qs[c][2 * mh + 1][2 * hh + part][tig];
      X[c][0] = x0.x; X[c][1] = x0.y; X[c][2] = x0.z; X[c][3] = x0.w;
      X[c][4] = x1.x; X[c][5] = x1.y; X[c][6] = x1.z; X[c][7] = x1.w;
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int ks = 4 * mh + q4;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t sp = __byte_perm(A[q4], B[q4], r ? 0x7632 : 0x5410);
        const int w = 2 * q4 + r;
        bq[ks][r] = split_mul(X[0][w], X[1][w], X[2][w], sp);
      }
    }
  }
}

// One 32-token packed tile on the tensor cores for the lane's head (tig).
__device__ __forceinline__ void mma_tile(const MmaSmem& s, const TileStage& st, int g, int tig,
                                         float scale_log2, float& m_run, float& lsum,
                                         float (&O)[8][4], float (&Z)[4]) {
  const int hh = g >> 1;
  const int part = g & 1;

  // ---- scores: S = codes x Q' (2 m-tiles of 16 tokens), beta = zK x q ----
  uint32_t bq[8][2];
  build_qprime(s, st, hh, part, tig, bq);
  float beta4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int mh = 0; mh < 2; ++mh) {
    const int m = 2 * tig + mh;
    const uint4 za = *reinterpret_cast<const uint4*>(&st.zk[kpad(8 * m)]);
    const uint4 zb = *reinterpret_cast<const uint4*>(&st.zk[kpad(8 * m + 4)]);
    const uint32_t A[4] = {za.x, za.y, za.z, za.w}, B[4] = {zb.x, zb.y, zb.z, zb.w};
    const uint4 b0 = s.qb[2 * mh][2 * hh + part][tig];
    const uint4 b1 = s.qb[2 * mh + 1][2 * hh + part][tig];
    const uint32_t QB[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint32_t z0 = __byte_perm(A[q4], B[q4], 0x5410);
      const uint32_t z1 = __byte_perm(A[q4], B[q4], 0x7632);
      mma16816(beta4, z0, z0, z1, z1, QB[2 * q4], QB[2 * q4 + 1]);
    }
  }
  const float beta = beta4[0] + beta4[1];

  float sc[4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint2 r0 = *reinterpret_cast<const uint2*>(&st.kc[(16 * mt + g) * 8 + 2 * tig]);
    const uint2 r1 = *reinterpret_cast<const uint2*>(&st.kc[(16 * mt + g + 8) * 8 + 2 * tig]);
    const uint32_t r0x10 = r0.x >> 10, r0y10 = r0.y >> 10, r1x10 = r1.x >> 10, r1y10 = r1.y >> 10;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#define KIVI_KSTEP(KS, I)                                                                  \
  {                                                                                        \
    const uint32_t wg = (KS) < 4 ? r0.x : r0.y, wgs = (KS) < 4 ? r0x10 : r0y10;           \
    const uint32_t w8 = (KS) < 4 ? r1.x : r1.y, w8s = (KS) < 4 ? r1x10 : r1y10;           \
    mma16816(acc, ext8<I>(wg, wgs), ext8<I>(w8, w8s), ext8<I + 1>(wg, wgs),                \
             ext8<I + 1>(w8, w8s), bq[KS][0], bq[KS][1]);                                  \
  }
    KIVI_KSTEP(0, 0) KIVI_KSTEP(1, 2) KIVI_KSTEP(2, 4) KIVI_KSTEP(3, 6)
    KIVI_KSTEP(4, 0) KIVI_KSTEP(5, 2) KIVI_KSTEP(6, 4) KIVI_KSTEP(7, 6)
#undef KIVI_KSTEP
    sc[2 * mt] = (acc[0] + acc[1] + beta) * scale_log2;      // token 16mt + g
    sc[2 * mt + 1] = (acc[2] + acc[3] + beta) * scale_log2;  // token 16mt + g + 8
  }

  // ---- online softmax of head tig over the 32 tokens (8 lanes share it) ----
  float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
  // The running max is raised (and the accumulators rescaled) only when a
  // score exceeds it by more than 8 in log2 units, so p <= 2^8 always.
  if (__any_sync(kFull, tmax > m_run + 8.0f)) {
    const float mnew = fmaxf(m_run, tmax);
    const float corr = fast_exp2(m_run - mnew);
    m_run = mnew;
    lsum *= corr;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) O[mt][i] *= corr;
#pragma unroll
    for (int i = 0; i < 4; ++i) Z[i] *= corr;
  }
  float p[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) p[r] = fast_exp2(sc[r] - m_run);  // token g + 8r
  lsum += (p[0] + p[1]) + (p[2] + p[3]);

  // ---- P for the value product: this lane needs head hh at tokens
  // 2tig + {0, 1} + 8r, held by lanes (2tig + delta, hh), value r ----
  float pv[2][4];
#pragma unroll
  for (int dl = 0; dl < 2; ++dl)
#pragma unroll
    for (int r = 0; r < 4; ++r) pv[dl][r] = __shfl_sync(kFull, p[r], 4 * (2 * tig + dl) + hh);

#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    uint32_t pa[2], Pp[4][2], az[2];
#pragma unroll
    for (int aa = 0; aa < 2; ++aa) {
      const int r = 2 * kk + aa;  // tokens 16kk + 8aa + 2tig + {0, 1}
      const uint32_t h = f2_to_h2(pv[0][r], pv[1][r]);
      const uint32_t l = f2_to_h2(pv[0][r] - h_lo(h), pv[1][r] - h_hi(h));
      // split_mul operands of this lane's part (see split_mul)
      pa[aa] = part ? l : h;
      const uint32_t pb = part ? h : 0u;
      const uint32_t pbn = pb ^ 0x80008000u;
      const int t0 = 16 * kk + 8 * aa + 2 * tig;
      const uint4 S = *reinterpret_cast<const uint4*>(&st.sv[2 * t0]);   // rows t0, t0 + 1
      const uint4 Zv = *reinterpret_cast<const uint4*>(&st.zv[2 * t0]);
      Pp[0][aa] = split_mul(pa[aa], pb, pbn, __byte_perm(S.x, S.z, 0x5410));
      Pp[1][aa] = split_mul(pa[aa], pb, pbn, __byte_perm(S.x, S.z, 0x7632));
      Pp[2][aa] = split_mul(pa[aa], pb, pbn, __byte_perm(S.y, S.w, 0x5410));
      Pp[3][aa] = split_mul(pa[aa], pb, pbn, __byte_perm(S.y, S.w, 0x7632));
      az[aa] = __byte_perm((g & 2) ? Zv.y : Zv.x, (g & 2) ? Zv.w : Zv.z, (g & 1) ? 0x7632 : 0x5410);
    }
    // z-term: rows = value groups (g & 3), columns = (head, part) of p
    mma16816(Z, az[0], az[0], az[1], az[1], pa[0], pa[1]);

    // value codes: interleaved word g of rows t0, t0 + 1 holds, per byte,
    // channels 4g..4g+3 of groups 0..3
    uint32_t u[2][2];  // [aa][groups 01 / 23]
#pragma unroll
    for (int aa = 0; aa < 2; ++aa) {
      const int t0 = 16 * kk + 8 * aa + 2 * tig;
      const uint32_t w0 = st.vc[t0 * 12 + g], w1 = st.vc[(t0 + 1) * 12 + g];
      u[aa][0] = __byte_perm(w0, w1, 0x5410);
      u[aa][1] = __byte_perm(w0, w1, 0x7632);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t x0 = u[0][half], x1 = u[1][half];
      const uint32_t x0s = x0 >> 10, x1s = x1 >> 10;
      // m-tiles 4*half + {0,1,2,3}: groups 2*half (bit pairs 0..3) and 2*half+1 (4..7)
#define KIVI_VTILE(MT, I, GP)                                                             \
  mma16816(O[MT], ext8<I>(x0, x0s), ext8<I + 1>(x0, x0s), ext8<I>(x1, x1s),               \
           ext8<I + 1>(x1, x1s), Pp[GP][0], Pp[GP][1]);
      if (half == 0) {
        KIVI_VTILE(0, 0, 0) KIVI_VTILE(1, 2, 0) KIVI_VTILE(2, 4, 1) KIVI_VTILE(3, 6, 1)
      } else {
        KIVI_VTILE(4, 0, 2) KIVI_VTILE(5, 2, 2) KIVI_VTILE(6, 4, 3) KIVI_VTILE(7, 6, 3)
      }
#undef KIVI_VTILE
    }
  }
}

// CTA prologue of the tensor-core path: q tables in fragment order.  Thread
// (head, tig, word) builds the pair words of both parts.
__device__ void build_q_tables(MmaSmem& s, const AttnArgs& a, int b, int j0, int nh) {
  for (int idx = threadIdx.x; idx < kNH * 4 * 16; idx += blockDim.x) {
    const int word = idx & 15;                // ks * 2 + r
    const int tig = (idx >> 4) & 3;
    const int hh = idx >> 6;
    const int ks = word >> 1, r = word & 1;
    const int m = 2 * tig + (ks >> 2);
    const int i = 2 * (ks & 3) + r;
    const float f = 1.0f / (float)(1 << (2 * pow4_exp(i)));
    float q2[2] = {0.0f, 0.0f};
    if (hh < nh)
#pragma unroll
      for (int half = 0; half < 2; ++half)
        q2[half] = load_q(a.q, ((long)b * a.Hq + j0 + hh) * kHeadDim + 16 * m + i + 8 * half, a.q_dtype);
    const uint32_t qh = f2_to_h2(q2[0], q2[1]);
    const uint32_t ql = f2_to_h2(q2[0] - h_lo(qh), q2[1] - h_hi(qh));
    const uint32_t sh = f2_to_h2(q2[0] * f, q2[1] * f);
    const uint32_t sl = f2_to_h2(q2[0] * f - h_lo(sh), q2[1] * f - h_hi(sh));
    const int quarter = word >> 2, wq = word & 3;
    // hi lane: (xa, xb, xbn) = (hi, 0, -0); lo lane: (lo, hi, -hi)
    reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh][tig])[wq] = sh;
    reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh][tig])[wq] = 0u;
    reinterpret_cast<uint32_t*>(&s.qs[2][quarter][2 * hh][tig])[wq] = 0x80008000u;
    reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh + 1][tig])[wq] = sl;
    reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh + 1][tig])[wq] = sh;
    reinterpret_cast<uint32_t*>(&s.qs[2][quarter][2 * hh + 1][tig])[wq] = sh ^ 0x80008000u;
    reinterpret_cast<uint32_t*>(&s.qb[quarter][2 * hh][tig])[wq] = qh;
    reinterpret_cast<uint32_t*>(&s.qb[quarter][2 * hh + 1][tig])[wq] = ql;
  }
}

// grid (splits, H * head_chunks, B), 128 threads.
template <int BITS>
__global__ void __launch_bounds__(128, kAttnCtasPerSm) attn_kernel(CacheView cv, AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];  // sizeof(SplitSmem)
  SplitSmem& sm = *reinterpret_cast<SplitSmem*>(smem_raw);
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
  const bool mma_path = (BITS == 2) && s > 0;
  float* mo = merge_area(sm, warp, mma_path);

  if (!mma_path) {
    // ---- CUDA cores: the tail split, or any split at 4 bits ----
    const int t_begin = s == 0 ? a.t_tail : (s - 1) * a.chunk;
    const int t_end = s == 0 ? a.l : min(a.t_tail, s * a.chunk);
    for (int i = threadIdx.x; i < kNH * kHeadDim; i += blockDim.x) {
      const int j = i / kHeadDim, d = i % kHeadDim;
      sm.v1.q[j][d] = j < nh ? load_q(a.q, ((long)b * a.Hq + j0 + j) * kHeadDim + d, a.q_dtype) * a.scale_log2
                             : 0.0f;
    }
    __syncthreads();
    float m[kNH], lsum[kNH], o[kNH][4];
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      m[j] = -INFINITY;
      lsum[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] = 0.0f;
    }
    if (t_begin < t_end) v1_tiles<BITS>(cv, a, sm, unit, t_begin, t_end, m, lsum, o);
#pragma unroll
    for (int j = 0; j < kNH; ++j) lsum[j] = warp_sum(lsum[j]);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        s_m[warp][j] = m[j];
        s_l[warp][j] = lsum[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kNH; ++j)
      *reinterpret_cast<float4*>(&mo[j * kHeadDim + 4 * lane]) = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
  } else {
    // ---- tensor cores: packed tiles [(s-1)*chunk, min(t_tail, s*chunk)) ----
    const int g = lane >> 2, tig = lane & 3;
    const int tile0 = (s - 1) * a.chunk / 32;
    const int tile1 = min(a.t_tail, s * a.chunk) / 32;
    const int n_mine = tile0 + warp < tile1 ? (tile1 - tile0 - warp + kWarps - 1) / kWarps : 0;
    TileStage* stages = sm.mma.st[warp];
    // start this warp's first tile copies before the CTA builds its q tables
    TileCopy tc = tile_copy_plan(cv, unit, tile0 + warp, lane);
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
      if (k < n_mine) issue_tile(tc, stages[k]);
      cp_async_commit();
      tile_copy_advance(tc);
    }
    build_q_tables(sm.mma, a, b, j0, nh);
    __syncthreads();
    float O[8][4], Z[4], m_run = -INFINITY, lsum = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) O[mt][i] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) Z[i] = 0.0f;
    int st_cur = 0, st_next = kStages - 1;
    for (int k = 0; k < n_mine; ++k) {
      if (k + kStages - 1 < n_mine) issue_tile(tc, stages[st_next]);
      cp_async_commit();
      tile_copy_advance(tc);
      cp_async_wait<kStages - 1>();
      __syncwarp();
      mma_tile(sm.mma, stages[st_cur], g, tig, a.scale_log2, m_run, lsum, O, Z);
      __syncwarp();
      st_cur = st_cur == kStages - 1 ? 0 : st_cur + 1;
      st_next = st_next == kStages - 1 ? 0 : st_next + 1;
    }
    cp_async_wait<0>();
    __syncwarp();
    // lane (g, tig) holds head tig: its partial sum over tokens g + 8r
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
    float* orow = mo + tig * kHeadDim;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int gp = mt >> 1, hm = mt & 1;
      const int i_lo = 4 * (gp & 1) + 2 * hm;
      const int ch = 32 * gp + 4 * g + 2 * hm;
      const float f_lo = 1.0f / (float)(1 << (2 * pow4_exp(i_lo)));
      const float f_hi = 1.0f / (float)(1 << (2 * pow4_exp(i_lo + 1)));
      orow[ch] = (O[mt][0] + O[mt][1]) * f_lo + zt[gp];
      orow[ch + 1] = (O[mt][2] + O[mt][3]) * f_hi + zt[gp];
    }
  }
  __syncthreads();

  // ---- merge the warps of this CTA into one partial per head ----
  const int d = threadIdx.x;
  for (int j = 0; j < nh; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][j]);
    float lt = 0.0f, ot = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = fast_exp2(s_m[w][j] - M);
        lt += e * s_l[w][j];
        ot += e * merge_area(sm, w, mma_path)[j * kHeadDim + d];
      }
    }
    const long pidx = ((long)b * a.Hq + j0 + j) * a.splits + s;
    a.ws_o[pidx * kHeadDim + d] = ot;
    if (d == 0) {
      a.ws_ml[pidx * 2] = M;
      a.ws_ml[pidx * 2 + 1] = lt;
    }
  }

  // ---- the last CTA of this (b, kv-head, head chunk) merges the splits ----
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* counter = a.counters + (long)b * gridDim.y + blockIdx.y;
    s_last = atomicAdd(counter, 1) == a.splits - 1;
    if (s_last) *counter = 0;  // every other CTA of the group has counted in
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // weights of the splits, one warp per head: e_s = 2^(m_s - M) / sum
  float* s_w = reinterpret_cast<float*>(&sm);  // [kNH][a.splits], the CTA's buffers are free now
  if (warp < nh) {
    const long base = ((long)b * a.Hq + j0 + warp) * a.splits;
    float M = -INFINITY;
    for (int sp = lane; sp < a.splits; sp += 32) M = fmaxf(M, __ldcg(a.ws_ml + (base + sp) * 2));
    M = warp_max(M);
    float den = 0.0f;
    for (int sp = lane; sp < a.splits; sp += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + (base + sp) * 2));
      const float e = ml.x == -INFINITY ? 0.0f : fast_exp2(ml.x - M);
      s_w[warp * a.splits + sp] = e;
      den += e * ml.y;
    }
    den = warp_sum(den);
    const float inv = 1.0f / den;
    for (int sp = lane; sp < a.splits; sp += 32) s_w[warp * a.splits + sp] *= inv;
  }
  __syncthreads();
  for (int j = 0; j < nh; ++j) {
    const long base = ((long)b * a.Hq + j0 + j) * a.splits;
    float num = 0.0f;
#pragma unroll 8
    for (int sp = 0; sp < a.splits; ++sp)
      num += s_w[j * a.splits + sp] * __ldcg(a.ws_o + (base + sp) * kHeadDim + d);
    const long oi = ((long)b * a.Hq + j0 + j) * kHeadDim + d;
    if (a.q_dtype == kF32) static_cast<float*>(a.out)[oi] = num;
    else if (a.q_dtype == kF16) static_cast<__half*>(a.out)[oi] = __float2half_rn(num);
    else static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(num);
  }
}

}  // namespace

template <int BITS>
cudaError_t launch_bits(const dim3& grid, const CacheView& cv, const AttnArgs& a, cudaStream_t st) {
  // The shared-memory opt-in is a per-device function attribute; setting it
  // on every call costs a host call only.
  const cudaError_t e = cudaFuncSetAttribute(attn_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(SplitSmem));
  if (e != cudaSuccess) return e;
  attn_kernel<BITS><<<grid, 128, sizeof(SplitSmem), st>>>(cv, a);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a, cudaStream_t st) {
  const int grp = a.Hq / cv.H;
  const int nhc = (grp + kNH - 1) / kNH;
  const dim3 grid(a.splits, cv.H * nhc, cv.B);
  return cv.bits == 2 ? launch_bits<2>(grid, cv, a, st) : launch_bits<4>(grid, cv, a, st);
}

}  // namespace kivi
