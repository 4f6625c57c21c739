// attention.cu -- decode attention over the packed KIVI cache.
//
// Decode step 2 of the chooblog KIVI review (§1.3): A = softmax(t_Q X_K^T),
// t_O = A X_V, scaled by 1/sqrt(D) as in the notebook "KIVI - 2-bit KV cache
// quantisation"; dequantization is fused into both products (review §3.2
// "System-Level": no separate dequantize pass).
//
// The context is split along the tokens (flash-decoding).  The tail
// [t_tail, l) -- the tokens whose keys or values are still fp16 in the
// residual rings, plus the partial value group before them -- runs on CUDA
// cores, in the first splits of every (batch, kv-head, head chunk) or after
// the tiles of its last packed split; the packed splits take the fully
// packed 32-token tiles [0, t_tail).  Partials are merged in the same
// launch: the CTA that finishes last in a group of up to kMergeGroup splits
// merges the group, and with more than one group the last group merges the
// groups; no CTA waits for another CTA of its launch.  (A launch that
// overlaps the launch before it waits, bounded, for the previous call on its
// workspace to publish a group's generation: see take_ticket.)  A CTA serves
// a chunk of up to eight query heads of one KV head, so every tile is decoded
// once for up to eight heads.
//
// Packed tiles (2, 3, 4 or 8 bits) run on the tensor cores (mma.sync
// m16n8k16, fp16 operands, fp32 accumulation).  Each warp streams its tiles
// through its own ring of staged tiles (one lane issues one bulk copy per
// tile, completion on an mbarrier) and keeps an online softmax per head:
//   scores  S[t, j] = sum_d c_td (q_jd s_d) + beta_j, beta_j = sum_d q_jd z_d
//           (beta per tile, for sixteen tiles per MMA in the split's prologue)
//   output  O[d, j] = sum_t c_td (p_jt s_t,g(d)) + sum_t p_jt z_t,g(d)
// The codes c enter the MMA as fp16 subnormals c * base^i * 2^-24 (the masked
// code bits are the whole encoding; base 4 at 2 and 3 bits, 16 at 4, 1 at 8).
// On the key side the fp32 factor q*s enters as an fp16 hi/lo pair (hi =
// fp16(x), lo = fp16(x - hi), together x to about 2^-22) in the 8 columns of
// the n=8 operand as (head, hi) and (head, lo), four heads per MMA: a single
// fp16 there would cost up to 2.1e-3 of relative output error on the
// streaming workload.  On the value side the weight p and p*s enter as one
// fp16 each, eight heads per MMA (at most 1.0e-3 on the same workloads; a
// CPU model of the rounding measured both); the weights' sums come out of the
// same product (ones in the z-term rows), so numerator and denominator use
// the same rounded p.  Each query head is first scaled by a power of two so
// that max |q| < 1, and a head's running max trails its scores by at most
// 0.5 (log2 units), so neither q*s nor p*s can overflow fp16.
#include <cuda_bf16.h>

#include <cstddef>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;
constexpr int kNH = kHeadChunk;  // query heads per CTA (one "head chunk")
constexpr uint32_t kOnesH2 = 0x3C003C00u;  // the fp16 pair {1, 1}
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



// ---------------------------------------------------------------------------
// Shared memory.

// q tables in MMA fragment order, one set per key block nb (query heads
// 4 nb .. 4 nb + 3).  Lane (g, tig) reads the 16 words of column g (head
// 4 nb + (g >> 1), part g & 1) for its tig, as four 16-byte quarters; the
// layout [quarter][column][tig] spreads the 8 lanes of a shared-memory phase
// over distinct banks.  Word w (k-step ks = w >> 1) of (column, tig) holds
// the channel pair of code position i:
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
  uint32_t sk[64];                        // key scales (the key zeros are not staged)
  uint32_t sv[64], zv[64];
  uint32_t outl[outlier_block_bytes(kMaxOutliers) / 4];  // outlier block, when the cache keeps outliers
};
constexpr int kMaxStages = 6;  // staged tiles per warp, at most
constexpr int kBetaTiles = 32;  // tiles of a warp whose beta = zK x q is held at once

// The packed splits' shared memory: per-warp rings of S staged tiles of
// `stride` bytes (the cache's tile size: a stage mirrors a tile byte for byte;
// S is chosen per launch to fill the CTA's share of the SM, see
// attn_stages), then this block.  q itself is staged for the table build in
// the stage buffers of stage 1, which no copy fills before the tables exist.
template <int NB>
struct PackedState {
  // q * base^-e(i) per column: one key block (NB = 1, columns (head, part)):
  // [0] / [1] the split_mul operands (xa, xb); two key blocks (NB = 2,
  // columns = heads): [0] / [1] the hi / lo part
  uint4 qs[2][4][8][4];
  uint4 qb[NB][4][8][4];                  // q hi / lo (words of a quarter in the order 0, 2, 1, 3)
  float qscale[kNH];                      // 2^E_j * softmax scale * log2(e)
  float qinv[kNH];                        // 2^-E_j: max |q_j| * 2^-E_j lies in [0.5, 1)
  // beta = zK x q of tile k of warp w at [w][k mod kBetaTiles][head hd]
  // (hd = tig with one key block, 2 tig + nb with two)
  float beta[kWarps][kBetaTiles][4 * NB];
  unsigned long long bar[kWarps][kMaxStages];
};

__host__ __device__ constexpr uint32_t packed_state_off(int S, uint32_t stride) {
  return ((uint32_t)kWarps * (uint32_t)S * stride + 15u) / 16u * 16u;
}

// A tail split: up to kTailTok tokens.  Its packed rows arrive as the whole
// code blocks of the (at most two) tiles involved (kpk, vpk, in the tiles'
// own layout), its fp16 residual rows as one or two runs of ring slots
// (kring, vring: token r of the split at row r), and the scale / zero blocks
// of those tiles whole (kg, vg), all by bulk copies on one mbarrier.
static_assert(kNH == 8, "the tail split keeps the heads of a channel / token in two float4");
template <int BITS>
struct TailSmem {
  float4 q8[kHeadDim][2];                 // q * scale * log2(e): the kNH heads of channel d
  __half kring[kTailTok][kHeadDim];       // fp16 key rows of the residual tokens
  __half vring[kTailTok][kHeadDim];       // fp16 value rows of the residual tokens
  uint8_t kpk[2][kGroup * kRowBytes<BITS>];  // key code blocks of the (at most two) tiles
  uint8_t vpk[2][kGroup * kRowBytes<BITS>];  // value code blocks
  uint32_t kg[2][2][64];                  // scale / zero of the (at most two) key groups
  uint32_t ko[2][outlier_block_bytes(kMaxOutliers) / 4];  // their outlier blocks
  uint32_t vg[2][2][64];                  // value scale / zero blocks of the (at most two) tiles
  float4 p8[kTailTok][2];                 // per token: scores, then weights, of the kNH heads
  float mh[kNH], lh[kNH];                 // per head: max and sum of the weights
  unsigned long long bar;                 // completion of the round's copies
};

enum Path { kPathMma = 1, kPathTail = 2 };

// The CTA's dynamic shared memory: the tail split's layout, or the packed
// splits' (stage rings, then PackedState), from the same base.
template <int BITS, int NB>
struct SmemView {
  unsigned char* base;
  int S;            // stages per warp
  uint32_t stride;  // bytes per stage

  __device__ __forceinline__ TileBuf<BITS>* ring(int w) const {
    return reinterpret_cast<TileBuf<BITS>*>(base + (size_t)w * S * stride);
  }
  __device__ __forceinline__ TileBuf<BITS>& stage(int w, int k) const {
    return *reinterpret_cast<TileBuf<BITS>*>(base + ((size_t)w * S + k) * stride);
  }
  __device__ __forceinline__ PackedState<NB>& ps() const {
    return *reinterpret_cast<PackedState<NB>*>(base + packed_state_off(S, stride));
  }
  __device__ __forceinline__ TailSmem<BITS>& tail() const { return *reinterpret_cast<TailSmem<BITS>*>(base); }
  // q * scale * log2(e) of the chunk's heads, [kNH][kHeadDim], after the
  // packed state: kept for the fp16 outlier key channels (present when the
  // cache keeps outlier channels, see attn_stages)
  __device__ __forceinline__ float* qo() const {
    return reinterpret_cast<float*>(base + packed_state_off(S, stride) + sizeof(PackedState<NB>));
  }
  // q of head j, staged for the tables: in stage 1 of warp j >> 1
  __device__ __forceinline__ float* qv(int j) const {
    return reinterpret_cast<float*>(base + ((size_t)(j >> 1) * S + 1) * stride + (j & 1) * 4 * kHeadDim);
  }
  // Per-warp merge area: [kNH][kHeadDim] floats inside buffers that the CTA
  // is done with (the warp's staged tiles, or the tail's rows).
  __device__ __forceinline__ float* merge_area(int warp, int path) const {
    if (path == kPathMma) return reinterpret_cast<float*>(base + (size_t)warp * S * stride);
    return reinterpret_cast<float*>(&tail().kring[0][0]) + warp * kNH * kHeadDim;
  }
};
static_assert(kWarps * kNH * kHeadDim * 4 <= 2 * kTailTok * kHeadDim, "tail merge areas");
// (a warp's merge area takes 4 KB: its S >= 2 stages of >= 2.75 KB hold it;
// two heads' q take 1 KB of its stage 1)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// mbarrier + bulk copy (one elected thread issues; the barrier's transaction
// count completes the phase when every byte has landed).
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// An mbarrier whose phases are all complete, invalidated before its shared
// memory is used for anything else.
__device__ __forceinline__ void mbar_inval(unsigned long long* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Orders this thread's earlier ordinary shared-memory accesses before later
// bulk copies into the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// The epoch protocol of overlapping calls on one workspace (thread 0): wait
// until the group's slot holds `want` (the previous call's epoch, published
// with release semantics after its last read of the group's slots), bounded
// like the staging waits; false when the wait gave up.  The call that
// publishes it belongs to an earlier launch on the stream, all of whose CTAs
// have started before any CTA of this one (a programmatic dependent starts
// only once every CTA of the launch before it has started), so the wait
// cannot hold up the CTA it waits for.
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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
constexpr unsigned kGenMask = 0xFFFFFFu;  // generations count modulo 2^24 (tickets wrap at 2^32)

// This launch's generation for group gid on its workspace, from a ticket:
// every launch that takes tickets (overlapping launches and decode steps'
// attention) adds kMaxSplits to the group's count (CTA 0 adds what the grid's
// other splits do not), and every CTA of such a launch has its ticket before
// any CTA of a later launch can start (the launch releases its dependents
// only after thread 0 has consumed the ticket), so ticket / kMaxSplits
// numbers these launches in stream order, CUDA graphs replayed included.
// Ordinary launches take none: they overlap no other launch, so what the
// count says stays true across them.  Thread 0 issues the atomic here and
// consumes it with ticket_gen.
__device__ __forceinline__ unsigned take_ticket(const AttnArgs& a, long gid) {
  const unsigned add = blockIdx.x == 0 ? (unsigned)(kMaxSplits - (int)gridDim.x + 1) : 1u;
  return atomicAdd(a.epochs + 2 * gid, add);
}
__device__ __forceinline__ unsigned ticket_gen(unsigned ticket) {
  return (ticket / (unsigned)kMaxSplits) & kGenMask;
}

__device__ bool epoch_wait(const unsigned* slot, unsigned want) {
  if (ld_acquire_u32(slot) == want) return true;
  const unsigned long long t0 = global_ns();
  while (ld_acquire_u32(slot) != want) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(256);
  }
  return true;
}

// The slot the epoch probe waits on: it stays 0, and the probe waits for 1.
__device__ unsigned g_probe_epoch;

__global__ void wait_probe_kernel(int* status) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (!mbar_wait(&bar, 0u)) atomicOr(status, 1);
    if (!epoch_wait(&g_probe_epoch, 1u)) atomicOr(status, 2);
  }
}

// ---------------------------------------------------------------------------
// A tail split on CUDA cores: tokens [c0, c0 + n), n <= kTailTok, of the tail
// [t_tail, l), staged in one round of copies (fp16 residual rows, packed rows
// and the key groups' scales / zeros), for the chunk's 4 NQ query heads.
// Scores: warp w takes tokens w, w + 4, ..., lane l channels 4l .. 4l + 3,
// and one transposing butterfly over the lanes sums the 4 NQ heads at once;
// the softmax of a head is one warp; values take one thread per channel.
// Keys and values of packed rows are dequantized as c * s + z with a single
// rounding, which equals the notebook's fl(fl(c * s) + z) because c * s is
// exact in fp32.  Leaves the partial of the CTA in warp 0's slots (the other
// warps' slots empty) and its output rows in `mo0` ([kNH][kHeadDim], inside
// the staged key rows).

// The codes of channels 4 lane .. 4 lane + 3 of packed key row `row` of a
// tile (the row's bytes as stored in the tile; channel e at bits
// (e * BITS) mod 8 of logical byte e * BITS / 8; at 3 bits the low two bits
// from the 2-bit plane, the high bit from its unit).
template <int BITS>
__device__ __forceinline__ void key_codes4(const uint8_t* rowp, int row, int lane, uint32_t (&c)[4]) {
  if constexpr (BITS == 2) {
    const uint32_t w = rowp[lane];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = (w >> (2 * i)) & 3u;
  } else if constexpr (BITS == 4) {
    const uint32_t w = reinterpret_cast<const uint16_t*>(rowp)[lane];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = (w >> (4 * i)) & 15u;
  } else if constexpr (BITS == 8) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(rowp + krow_byte<8>(row, 4 * lane));
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = (w >> (8 * i)) & 255u;
  } else {
    const uint32_t w = rowp[lane];
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(rowp);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;  // the channel
      const uint32_t hi =
          (rw[kHiPlane3 / 4 + ((e >> 4) & 3)] >> (16 * ((e >> 3) & 1) + hi_bit3(e >> 6, e & 7))) & 1u;
      c[i] = ((w >> (2 * i)) & 3u) | (hi << 2);
    }
  }
}

// Sum of v[0..H) over the 32 lanes, H heads at once: each butterfly level
// halves the values a lane carries (the lanes with bit `o` set keep the upper
// half), then plain levels finish the sums.  Every lane of a block of 32 / H
// lanes ends with the total of head `head`.
template <int H>
__device__ __forceinline__ float reduce_heads(const float (&v)[H], int lane, int& head) {
  float cur[H];
#pragma unroll
  for (int i = 0; i < H; ++i) cur[i] = v[i];
  head = 0;
  int o = 16;
#pragma unroll
  for (int half = H / 2; half >= 1; half >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? cur[i + half] : cur[i];
      const float send = up ? cur[i] : cur[i + half];
      cur[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
    head += up ? half : 0;
    o >>= 1;
  }
#pragma unroll
  for (; o > 0; o >>= 1) cur[0] += __shfl_xor_sync(kFull, cur[0], o);
  return cur[0];
}

template <int BITS, int NQ>
__device__ __noinline__ void tail_split(const CacheView& cv, const AttnArgs& a, const SeqPlan p, TailSmem<BITS>& ts,
                                        float* mo0, long unit, int b, int j0, int nh, int c0, uint32_t round,
                                        float (&s_m)[kWarps][kNH], float (&s_l)[kWarps][kNH]) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;  // packed row bytes
  constexpr int H = 4 * NQ;                // heads of this tail
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = min(kTailTok, p.l - c0);
  const int nk = max(0, min(n, p.nq_k - c0));  // rows [0, nk) hold packed keys
  const int nv = max(0, min(n, p.nq_v - c0));  // rows [0, nv) hold packed values
  const int ngk = (nk + kGroup - 1) / kGroup, ngv = (nv + kGroup - 1) / kGroup;
  const int tile0 = c0 / kGroup;  // c0 is a multiple of 32: packed rows span at most two tiles

  // ---- stage the round with bulk copies (thread 0), and q ----
  if (tid == 0) {
    if (round == 0) {
      mbar_init(&ts.bar, 1);
      mbar_fence_init();
    }
    fence_proxy_async();  // the buffers were last used by ordinary loads and stores
    const int ob = outlier_block_bytes(cv.n_out);
    const int wk = n - nk, wv = n - nv;  // residual rows of keys / values
    const int sk0 = (int)((c0 + nk) % cv.W), sv0 = (int)((c0 + nv) % cv.W);
    const int k1 = min(wk, cv.W - sk0), v1 = min(wv, cv.W - sv0);  // first runs of ring slots
    const uint32_t bytes = (uint32_t)(ngk * (kGroup * RB + 4 * kHeadDim + ob) + ngv * (kGroup * RB + 4 * kHeadDim) +
                                      (wk + wv) * 2 * kHeadDim);
    mbar_expect_tx(&ts.bar, bytes);
    for (int gi = 0; gi < ngk; ++gi) {
      const uint8_t* tile = tile_at<BITS>(cv, unit, tile0 + gi);
      bulk_g2s(ts.kpk[gi], tile + kOffKc<BITS>, kGroup * RB, &ts.bar);
      bulk_g2s(ts.kg[gi][0], tile + kOffSk<BITS>, 2 * kHeadDim, &ts.bar);  // scales
      bulk_g2s(ts.kg[gi][1], tile + kOffZk, 2 * kHeadDim, &ts.bar);        // zeros
      if (ob) bulk_g2s(ts.ko[gi], tile + kTileBytes<BITS>, ob, &ts.bar);
    }
    for (int gi = 0; gi < ngv; ++gi) {
      const uint8_t* tile = tile_at<BITS>(cv, unit, tile0 + gi);
      bulk_g2s(ts.vpk[gi], tile + kOffVc<BITS>, kGroup * RB, &ts.bar);
      bulk_g2s(ts.vg[gi], tile + kOffSv<BITS>, 4 * kHeadDim, &ts.bar);
    }
    const __half* rk = cv.ring_k + unit * cv.W * kHeadDim;
    const __half* rv = cv.ring_v + unit * cv.W * kHeadDim;
    if (k1 > 0) bulk_g2s(ts.kring[nk], rk + (long)sk0 * kHeadDim, k1 * 2 * kHeadDim, &ts.bar);
    if (wk > k1) bulk_g2s(ts.kring[nk + k1], rk, (wk - k1) * 2 * kHeadDim, &ts.bar);
    if (v1 > 0) bulk_g2s(ts.vring[nv], rv + (long)sv0 * kHeadDim, v1 * 2 * kHeadDim, &ts.bar);
    if (wv > v1) bulk_g2s(ts.vring[nv + v1], rv, (wv - v1) * 2 * kHeadDim, &ts.bar);
  }
  {
    float qj[kNH];
#pragma unroll
    for (int j = 0; j < kNH; ++j)
      qj[j] = j < nh ? load_q(a.q, ((long)b * a.Hq + j0 + j) * kHeadDim + tid, a.q_dtype) * a.scale_log2 : 0.0f;
    ts.q8[tid][0] = make_float4(qj[0], qj[1], qj[2], qj[3]);
    ts.q8[tid][1] = make_float4(qj[4], qj[5], qj[6], qj[7]);
  }
  __syncthreads();  // q staged; the barrier initialized before anyone waits on it
  if (!mbar_wait(&ts.bar, round & 1u) && tid == 0) atomicOr(a.status, 1);

  // ---- scores: warp w takes tokens w, w + 4, ... (two at a time); lane l
  //      channels 4l..4l+3 ----
  {
    float qr[4][H];  // q of this lane's channels, the tail's heads
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq) {
        const float4 v = ts.q8[4 * lane + c][nq];
        qr[c][4 * nq] = v.x;
        qr[c][4 * nq + 1] = v.y;
        qr[c][4 * nq + 2] = v.z;
        qr[c][4 * nq + 3] = v.w;
      }
    // scales / zeros of this lane's channels in the (at most two) key groups
    float ks_[2][4], kz_[2][4];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int pos = kscale_pos<BITS>(4 * lane + c);
        ks_[gi][c] = gi < ngk ? __half2float(reinterpret_cast<const __half*>(ts.kg[gi][0])[pos]) : 0.0f;
        kz_[gi][c] = gi < ngk ? __half2float(reinterpret_cast<const __half*>(ts.kg[gi][1])[pos]) : 0.0f;
      }
    auto score = [&](int r, float (&acc)[H]) {
      float kx[4];
      if (r < nk) {
        uint32_t cd[4];
        key_codes4<BITS>(ts.kpk[r >> 5] + (r & 31) * RB, r & 31, lane, cd);
        const int gi = r >> 5;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          kx[c] = fmaf(__uint_as_float(cd[c] | 0x4B000000u) - 8388608.0f, gi ? ks_[1][c] : ks_[0][c],
                       gi ? kz_[1][c] : kz_[0][c]);
      } else {
        const uint2 h4 = *reinterpret_cast<const uint2*>(&ts.kring[r][4 * lane]);
        kx[0] = h_lo(h4.x);
        kx[1] = h_hi(h4.x);
        kx[2] = h_lo(h4.y);
        kx[3] = h_hi(h4.y);
      }
#pragma unroll
      for (int j = 0; j < H; ++j) {
        acc[j] = kx[0] * qr[0][j];
#pragma unroll
        for (int c = 1; c < 4; ++c) acc[j] = fmaf(kx[c], qr[c][j], acc[j]);
      }
      if (lane == 0 && r < nk && cv.n_out > 0) {
        // the group's fp16 outlier channels (their packed codes decode to 0)
        const uint32_t iw = ts.ko[r >> 5][0];
        const __half* ov = reinterpret_cast<const __half*>(&ts.ko[r >> 5][4]);
        for (int o = 0; o < cv.n_out; ++o) {
          const float x = __half2float(ov[(r & 31) * cv.n_out + o]);
          const float* qo = reinterpret_cast<const float*>(&ts.q8[(iw >> (8 * o)) & 0xffu][0]);
#pragma unroll
          for (int j = 0; j < H; ++j) acc[j] = fmaf(x, qo[j], acc[j]);
        }
      }
    };
#pragma unroll 1
    for (int r = warp; r < n; r += 2 * kWarps) {
      const int r1 = r + kWarps < n ? r + kWarps : r;  // a second token (or the first again)
      float acc0[H], acc1[H];
      score(r, acc0);
      score(r1, acc1);
      int head;
      const float s0 = reduce_heads<H>(acc0, lane, head);
      const float s1 = reduce_heads<H>(acc1, lane, head);
      if ((lane & (32 / H - 1)) == 0) {
        reinterpret_cast<float*>(ts.p8)[r * kNH + head] = s0;
        reinterpret_cast<float*>(ts.p8)[r1 * kNH + head] = s1;
      }
    }
  }
  __syncthreads();

  // ---- softmax of heads `warp` (and `warp` + 4) over the round ----
#pragma unroll
  for (int hh = 0; hh < NQ; ++hh) {
    const int j = warp + kWarps * hh;
    float* pj = reinterpret_cast<float*>(ts.p8) + j;  // [token][kNH]
    const float x0 = lane < n ? pj[kNH * lane] : -INFINITY;
    const float x1 = lane + 32 < n ? pj[kNH * (lane + 32)] : -INFINITY;
    const float mx = warp_max(fmaxf(x0, x1));
    const float e0 = lane < n ? fast_exp2(x0 - mx) : 0.0f;
    const float e1 = lane + 32 < n ? fast_exp2(x1 - mx) : 0.0f;
    pj[kNH * lane] = e0;
    pj[kNH * (lane + 32)] = e1;
    const float sum = warp_sum(e0 + e1);
    if (lane == 0) {
      ts.mh[j] = mx;
      ts.lh[j] = sum;
    }
  }
  __syncthreads();

  // ---- values: thread d accumulates channel d of the tail's heads ----
  const int d = tid;
  const int vpos = v_unit_pos(d >> 2);
  const int vsh = BITS * (d & 3);
  float o[H];
#pragma unroll
  for (int j = 0; j < H; ++j) o[j] = 0.0f;
#pragma unroll 2
  for (int r = 0; r < n; ++r) {
    float vx;
    if (r < nv) {
      const uint8_t* row = ts.vpk[r >> 5] + (r & 31) * RB;
      uint32_t cb;
      if constexpr (BITS == 2) cb = row[vpos];
      else if constexpr (BITS == 3) cb = row[vpos] | ((uint32_t)*reinterpret_cast<const uint16_t*>(row + kHiPlane3 + 2 * ((d & 31) >> 2)) << 8);
      else if constexpr (BITS == 4) cb = *reinterpret_cast<const uint16_t*>(row + 2 * vpos);
      else cb = *reinterpret_cast<const uint32_t*>(row + vrow_byte<8>(r & 31, 4 * vpos));
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
      vx = __half2float(ts.vring[r][d]);
    }
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
      const float4 pr = ts.p8[r][nq];
      o[4 * nq] = fmaf(pr.x, vx, o[4 * nq]);
      o[4 * nq + 1] = fmaf(pr.y, vx, o[4 * nq + 1]);
      o[4 * nq + 2] = fmaf(pr.z, vx, o[4 * nq + 2]);
      o[4 * nq + 3] = fmaf(pr.w, vx, o[4 * nq + 3]);
    }
  }
  __syncthreads();  // every thread is done with the staged rows (the merge area)

#pragma unroll
  for (int j = 0; j < H; ++j) mo0[j * kHeadDim + d] = o[j];
  if (lane < kNH) {
    s_m[warp][lane] = warp == 0 && lane < H ? ts.mh[lane] : -INFINITY;
    s_l[warp][lane] = warp == 0 && lane < H ? ts.lh[lane] : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Tensor-core path (packed tiles).

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A x B (no accumulator input: the C operand is the literal zero, which
// the tensor instruction reads as the zero register), or D += A x B.
template <bool kFirst>
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  if constexpr (kFirst) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f), "f"(0.0f), "f"(0.0f), "f"(0.0f));
  } else {
    mma16816(d, a0, a1, a2, a3, b0, b1);
  }
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
// that later tiles rarely raise it again (on the Llama-3-8B decode shape
// about 4% of the tiles after the first raise it, against 37% with a slack
// of 1).  The weights then lie in (0, 2^0.5], and right after a raise the
// largest is 2^-3: fp16 keeps its full relative precision for p * s.
constexpr float kLazySlack = 3.0f;

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

// Q' = q * sK of one key group as MMA B fragments for column g of this lane,
// in the order of the q tables: one key block, head g >> 1, part g & 1 (one
// fp16 of the pair per lane); two key blocks, head g, both parts (bq[0] hi,
// bq[1] lo).  The q table is pre-scaled by base^-e(i) to cancel the power
// that the code extraction leaves in the A operand.
template <int BITS, int NB>
__device__ __forceinline__ void build_qprime(const PackedState<NB>& ws, const uint32_t* sk, int g, int tig,
                                             uint32_t (&bq)[NB][8][2]) {
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
        const uint32_t sp = P[word_pos<BITS>(w)];
        if constexpr (NB == 1) {
          bq[0][w >> 1][w & 1] = split_mul(X0[wq], X1[wq], sp);
        } else {
          // both parts of head g: hi = fp16(qh s), lo = fp16(ql s + (qh s - hi))
          const uint32_t hi = hmul2u(X0[wq], sp);
          bq[0][w >> 1][w & 1] = hi;
          bq[NB - 1][w >> 1][w & 1] = hfma2u(X1[wq], sp, hfms2u(X0[wq], sp, hi));
        }
      }
    }
  }
}

// Row of the score product: m-tile row g of a 16-token m-tile takes token
// tau(g) of it and row g + 8 token tau(g) + 4, so that the lane holding the
// scores of rows (g, g + 8) holds exactly the token pair (t, t + 4) that one
// B-fragment register of the value product takes.
__device__ __forceinline__ int score_row(int g) { return (g & 3) + 8 * (g >> 2); }

// Scores of one staged 32-token tile: lane (g, tig) gets head hd(nb) at
// tokens 16 (r >> 1) + score_row(g) + 4 (r & 1) in sc[nb][r] (log2 units),
// less mb[nb], where hd(nb) = tig with one key block and 2 tig + nb with two;
// ks = 2^E * scale * log2(e) of that head.
template <int BITS, int NB>
__device__ __forceinline__ void key_scores(const PackedState<NB>& ws, const TileBuf<BITS>& tb, int g, int tig,
                                           const float (&ks)[NB], const float (&mb)[NB], int n_out,
                                           const float* qo, const float* brow, float (&sc)[NB][4]) {
  constexpr int RW = 4 * BITS;  // 32-bit words per code row
  float kbm[NB];  // beta * ks - mb, the score offset of the tile (beta from brow, see beta_mma)
  if constexpr (NB == 1) {
    kbm[0] = fmaf(brow[tig], ks[0], -mb[0]);
  } else {
    const float2 b2 = *reinterpret_cast<const float2*>(brow + 2 * tig);
    kbm[0] = fmaf(b2.x, ks[0], -mb[0]);
    kbm[NB - 1] = fmaf(b2.y, ks[NB - 1], -mb[NB - 1]);
  }

  // ---- scores S = codes x Q' + beta ----
  uint32_t bq[NB][8][2];
  build_qprime<BITS, NB>(ws, tb.sk, g, tig, bq);
  const int tr = score_row(g);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + tr, r1 = r0 + 4;  // the key rows of m-tile rows g and g + 8
    const uint32_t* rg = tb.kc + r0 * RW;
    const uint32_t* r8 = tb.kc + r1 * RW;
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
        const uint4 a0 = reinterpret_cast<const uint4*>(rg)[krow_chunk<8>(r0, 2 * tig + h)];
        const uint4 a1 = reinterpret_cast<const uint4*>(r8)[krow_chunk<8>(r1, 2 * tig + h)];
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
    float acc[NB][4];  // written first by k-step 0 (no accumulator input)
#define KIVI_MMA_NB(KS, A0, A1, A2, A3)                                                      \
  {                                                                                          \
    const uint32_t a0_ = (A0), a1_ = (A1), a2_ = (A2), a3_ = (A3);                           \
    _Pragma("unroll") for (int nb = 0; nb < NB; ++nb)                                        \
        mma_acc<(KS) == 0>(acc[nb], a0_, a1_, a2_, a3_, bq[nb][KS][0], bq[nb][KS][1]);       \
  }
    if constexpr (BITS == 3) {
      const uint32_t hg0 = rg[kHiPlane3 / 4 + tig], h80 = r8[kHiPlane3 / 4 + tig];
      const uint32_t hg1 = swap_half_bytes(hg0), h81 = swap_half_bytes(h80);
      // high sources of word j (set j): h, h >> 1
      const uint32_t hg[2] = {hg0, hg1}, h8[2] = {h80, h81};
      const uint32_t hgs[2] = {hg0 >> 1, hg1 >> 1}, h8s[2] = {h80 >> 1, h81 >> 1};
#define KIVI_KSTEP3(KS, I)                                                                    \
  KIVI_MMA_NB(KS, ext3<I>(wg[(KS) >> 2], sg[(KS) >> 2], hg[(KS) >> 2], hgs[(KS) >> 2]),       \
              ext3<I>(w8[(KS) >> 2], s8[(KS) >> 2], h8[(KS) >> 2], h8s[(KS) >> 2]),           \
              ext3<I + 1>(wg[(KS) >> 2], sg[(KS) >> 2], hg[(KS) >> 2], hgs[(KS) >> 2]),       \
              ext3<I + 1>(w8[(KS) >> 2], s8[(KS) >> 2], h8[(KS) >> 2], h8s[(KS) >> 2]))
      KIVI_KSTEP3(0, 0) KIVI_KSTEP3(1, 2) KIVI_KSTEP3(2, 4) KIVI_KSTEP3(3, 6)
      KIVI_KSTEP3(4, 0) KIVI_KSTEP3(5, 2) KIVI_KSTEP3(6, 4) KIVI_KSTEP3(7, 6)
#undef KIVI_KSTEP3
    } else if constexpr (BITS == 2) {
#define KIVI_KSTEP(KS, I)                                                                     \
  KIVI_MMA_NB(KS, (ext<2, I>(wg[(KS) >> 2], sg[(KS) >> 2])), (ext<2, I>(w8[(KS) >> 2], s8[(KS) >> 2])), \
              (ext<2, I + 1>(wg[(KS) >> 2], sg[(KS) >> 2])), (ext<2, I + 1>(w8[(KS) >> 2], s8[(KS) >> 2])))
      KIVI_KSTEP(0, 0) KIVI_KSTEP(1, 2) KIVI_KSTEP(2, 4) KIVI_KSTEP(3, 6)
      KIVI_KSTEP(4, 0) KIVI_KSTEP(5, 2) KIVI_KSTEP(6, 4) KIVI_KSTEP(7, 6)
#undef KIVI_KSTEP
    } else if constexpr (BITS == 4) {
#define KIVI_KSTEP(KS, I)                                                                     \
  KIVI_MMA_NB(KS, (ext<4, I>(wg[(KS) >> 1], sg[(KS) >> 1])), (ext<4, I>(w8[(KS) >> 1], s8[(KS) >> 1])), \
              (ext<4, I + 1>(wg[(KS) >> 1], sg[(KS) >> 1])), (ext<4, I + 1>(w8[(KS) >> 1], s8[(KS) >> 1])))
      KIVI_KSTEP(0, 0) KIVI_KSTEP(1, 2) KIVI_KSTEP(2, 0) KIVI_KSTEP(3, 2)
      KIVI_KSTEP(4, 0) KIVI_KSTEP(5, 2) KIVI_KSTEP(6, 0) KIVI_KSTEP(7, 2)
#undef KIVI_KSTEP
    } else {
      // k-step ks: word ks (channels 4m .. 4m + 3, m = 8 tig + ks), bytes 0 / 2
      // then bytes 1 / 3 of each half
#define KIVI_KSTEP8(KS)                                                                       \
  KIVI_MMA_NB(KS, (ext<8, 0>(wg[KS], sg[KS])), (ext<8, 0>(w8[KS], s8[KS])), (ext<8, 1>(wg[KS], sg[KS])), \
              (ext<8, 1>(w8[KS], s8[KS])))
      KIVI_KSTEP8(0) KIVI_KSTEP8(1) KIVI_KSTEP8(2) KIVI_KSTEP8(3)
      KIVI_KSTEP8(4) KIVI_KSTEP8(5) KIVI_KSTEP8(6) KIVI_KSTEP8(7)
#undef KIVI_KSTEP8
    }
#undef KIVI_MMA_NB
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float k24 = ks[nb] * kTwo24;
      const float s0 = NB == 1 ? acc[0][0] + acc[0][1] : acc[0][nb] + acc[NB - 1][nb];
      const float s1 = NB == 1 ? acc[0][2] + acc[0][3] : acc[0][2 + nb] + acc[NB - 1][2 + nb];
      sc[nb][2 * mt] = fmaf(s0, k24, kbm[nb]);      // token r0
      sc[nb][2 * mt + 1] = fmaf(s1, k24, kbm[nb]);  // token r0 + 4
    }
  }
  if (n_out > 0) {
    // fp16 outlier channels (their codes, scales and zeros are 0 above)
    const uint32_t iw = tb.outl[0];
    const __half* ov = reinterpret_cast<const __half*>(&tb.outl[4]);  // [32 tokens][n_out]
#pragma unroll
    for (int o = 0; o < kMaxOutliers; ++o)
      if (o < n_out) {
        const int ch = (iw >> (8 * o)) & 0xffu;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const float qx = qo[(NB == 1 ? tig : 2 * tig + nb) * kHeadDim + ch];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int t = 16 * (r >> 1) + tr + 4 * (r & 1);
            sc[nb][r] = fmaf(qx, __half2float(ov[t * n_out + o]), sc[nb][r]);
          }
        }
      }
  }
}

// Online softmax over one tile's scores (lane (g, tig) holds head hd(nb) of
// key_scores at four tokens; 8 lanes share a head): when a score exceeds a head's
// running max by more than kLazyMax, the max is raised to the tile max plus
// kLazySlack and what the earlier tiles left in O and Z is rescaled.  The
// weights p = 2^(S - max) <= 2^kLazyMax are rounded to fp16 pairs and moved
// to the value product's B fragments: lane (g, tig) gets head g at tokens
// (16 kk + 8 aa + tig, + 4) in pb[kk][aa].
// The scores arrive as x = S - mb with mb = m_run, or 0 while m_run is still
// -inf (before the first tile).
template <int NB>
__device__ __forceinline__ void softmax_p(float (&x)[NB][4], int g, int tig, float (&m_run)[NB],
                                          float (&O)[8][4], float (&Z)[4], uint32_t (&pb)[2][2]) {
  float mx = -INFINITY;
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int r = 0; r < 4; ++r) mx = fmaxf(mx, x[nb][r]);
  bool first = false;
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) first |= m_run[nb] == -INFINITY;
  if (__any_sync(kFull, first || mx > kLazyMax)) {
    float corr[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float mb = m_run[nb] == -INFINITY ? 0.0f : m_run[nb];
      float t = fmaxf(fmaxf(x[nb][0], x[nb][1]), fmaxf(x[nb][2], x[nb][3]));
      t = fmaxf(t, __shfl_xor_sync(kFull, t, 4));
      t = fmaxf(t, __shfl_xor_sync(kFull, t, 8));
      t = fmaxf(t, __shfl_xor_sync(kFull, t, 16));
      t += mb;  // the tile max of head 4 nb + tig
      const float mnew = t > m_run[nb] + kLazyMax ? t + kLazySlack : m_run[nb];
      corr[nb] = fast_exp2(m_run[nb] - mnew);  // 0 on the first tile
      m_run[nb] = mnew;
      const float dm = mb - mnew;
#pragma unroll
      for (int r = 0; r < 4; ++r) x[nb][r] += dm;
    }
    // the O and Z columns of this lane are heads 2 tig and 2 tig + 1: with
    // two key blocks its own heads; with one, heads held by lanes (2 tig) & 3
    // and (2 tig + 1) & 3 (the columns of heads 4..7 are unused)
    float cA, cB;
    if constexpr (NB == 2) {
      cA = corr[0];
      cB = corr[NB - 1];
    } else {
      cA = __shfl_sync(kFull, corr[0], (2 * tig) & 3);
      cB = __shfl_sync(kFull, corr[0], (2 * tig + 1) & 3);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      O[mt][0] *= cA;
      O[mt][1] *= cB;
      O[mt][2] *= cA;
      O[mt][3] *= cB;
    }
    Z[0] *= cA;
    Z[1] *= cB;
    Z[2] *= cA;
    Z[3] *= cB;
  }
  uint32_t P2[NB][2];  // fp16 weights of tokens (16 mt + score_row(g), + 4)
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
      P2[nb][mt] = f2_to_h2(fast_exp2(x[nb][2 * mt]), fast_exp2(x[nb][2 * mt + 1]));
  // token 16 kk + 8 aa + tig is row score_row^-1(8 aa + tig) = tig + 4 aa of
  // m-tile kk; head g is held by lane (.., g & 3) (one key block, block 0)
  // or lane (.., g >> 1), block g & 1 (two key blocks)
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
#pragma unroll
    for (int aa = 0; aa < 2; ++aa) {
      const int src = 4 * (tig + 4 * aa) + (NB == 2 ? g >> 1 : g & 3);
      const uint32_t v0 = __shfl_sync(kFull, P2[0][kk], src);
      if constexpr (NB == 2) {
        const uint32_t v1 = __shfl_sync(kFull, P2[NB - 1][kk], src);
        pb[kk][aa] = (g & 1) ? v1 : v0;
      } else {
        pb[kk][aa] = v0;  // columns 4..7 repeat heads 0..3 and are not used
      }
    }
}

// Values of one staged tile: O += codes^T x (p * sV), Z += [zV; 1]^T x p,
// with the fp16 weights pb of the tile (column g = head g).  The k rows
// (2tig, 2tig+1) of k-step kk hold tokens t0 = 16kk + tig and t0 + 4, rows
// (2tig+8, 2tig+9) tokens t0 + 8 and t0 + 12.  M-tile 2gp + hm covers value
// group gp: row g is channel 32gp + 4g + 2hm, row g + 8 the next channel.
// Row g of the z-term product is value group g & 3, row g + 8 all ones, so
// Z[2], Z[3] accumulate the sums of the weights of this lane's heads.
template <int BITS>
__device__ __forceinline__ void value_acc(const TileBuf<BITS>& tb, const uint32_t (&pb)[2][2], int g, int tig,
                                          float (&O)[8][4], float (&Z)[4]) {
  constexpr int RW = 4 * BITS;  // 32-bit words per code row
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    // u[aa][gp]: the codes of channels 4g..4g+3 of group gp for tokens (t0,
    // t0 + 4), as the two 16-bit halves (2 bits: a byte per group, two groups
    // per word)
    uint32_t Pp[4][2], az[2], u[2][4];
    uint32_t v8a[2][4], v8b[2][4];  // 8 bits: unit words of groups 0..3 of tokens t0 and t0 + 4
    uint32_t hv[2][2];              // 3 bits: high units of tokens (t0, t0 + 4), groups 0/1 and 2/3
#pragma unroll
    for (int aa = 0; aa < 2; ++aa) {
      const int t0 = 16 * kk + 8 * aa + tig;  // tokens t0, t0 + 4
      // the scale / zero words of token pair (t0, t0 + 4) (see vscale_pos)
      const int pw = 4 * (4 * (2 * kk + aa) + tig);
      const uint4 S = *reinterpret_cast<const uint4*>(tb.sv + pw);  // groups 0..3
      Pp[0][aa] = hmul2u(pb[kk][aa], S.x);
      Pp[1][aa] = hmul2u(pb[kk][aa], S.y);
      Pp[2][aa] = hmul2u(pb[kk][aa], S.z);
      Pp[3][aa] = hmul2u(pb[kk][aa], S.w);
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
    // z-term and weight sums: rows g = value group g & 3, rows g + 8 = ones
    mma16816(Z, az[0], kOnesH2, az[1], kOnesH2, pb[kk][0], pb[kk][1]);
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
// (warp w takes heads w and w + 4), then the tables in fragment order.
// Thread (block, head, tig, word) builds the pair words of both parts.
static_assert(kNH == 2 * kWarps, "warp w loads and scales heads w and w + 4");

// Channels 4 lane .. 4 lane + 3 of the CTA's heads `warp` (v[0..3]) and
// `warp` + 4 (v[4..7]), zeros past the last head.  Issued before the first
// tile copies, so that the load does not queue behind them.
__device__ __forceinline__ void load_q8(const AttnArgs& a, int b, int j0, int nh, float (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = warp + kWarps * hh;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[4 * hh + i] = j < nh ? load_q(a.q, ((long)b * a.Hq + j0 + j) * kHeadDim + 4 * lane + i, a.q_dtype) : 0.0f;
  }
}

template <int BITS, int NB>
__device__ void build_q_tables(const SmemView<BITS, NB>& sv, const AttnArgs& a, const float (&v)[8], bool keep_q) {
  PackedState<NB>& s = sv.ps();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = warp + kWarps * hh;
    const float* vj = v + 4 * hh;
    *reinterpret_cast<float4*>(sv.qv(j) + 4 * lane) = make_float4(vj[0], vj[1], vj[2], vj[3]);
    if (keep_q) {
      const float sl = a.scale_log2;
      *reinterpret_cast<float4*>(sv.qo() + j * kHeadDim + 4 * lane) =
          make_float4(vj[0] * sl, vj[1] * sl, vj[2] * sl, vj[3] * sl);
    }
    const float amax = warp_max(fmaxf(fmaxf(fabsf(vj[0]), fabsf(vj[1])), fmaxf(fabsf(vj[2]), fabsf(vj[3]))));
    if (lane == 0) {
      const int be = (int)((__float_as_uint(amax) >> 23) & 0xffu);
      // amax in [2^(be-127), 2^(be-126)) for normal amax; a subnormal amax is
      // below 2^-126, a zero row keeps E = 0
      const int E = amax == 0.0f ? 0 : (be == 0 ? -126 : be - 126);
      s.qinv[j] = ldexpf(1.0f, -E);  // exact: a power of two (subnormal for E > 126)
      s.qscale[j] = ldexpf(a.scale_log2, E);
    }
  }
  __syncthreads();
  // one key block: heads 0..3, each in columns (2 hh, 2 hh + 1) as (hi, lo);
  // two key blocks: heads 0..7 in columns 0..7, one table per part
  for (int idx = threadIdx.x; idx < NB * 4 * 4 * 16; idx += blockDim.x) {
    const int word = idx & 15;                // ks * 2 + r
    const int tig = (idx >> 4) & 3;
    const int j = idx >> 6;                   // the head
    const int hh = j & 3;
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
    const float q0 = sv.qv(j)[c0] * s.qinv[j], q1 = sv.qv(j)[c1] * s.qinv[j];  // exact scalings
    const uint32_t qh = f2_to_h2(q0, q1);
    const uint32_t ql = f2_to_h2(q0 - h_lo(qh), q1 - h_hi(qh));
    const uint32_t sh = f2_to_h2(q0 * f, q1 * f);
    const uint32_t sl = f2_to_h2(q0 * f - h_lo(sh), q1 * f - h_hi(sh));
    const int quarter = word >> 2, wq = word & 3;
    // the beta MMAs take words (0, 2) and (1, 3) of a quarter as B pairs
    const int wb = wq == 1 ? 2 : (wq == 2 ? 1 : wq);
    if constexpr (NB == 1) {
      // hi lane: (xa, xb) = (hi, 0); lo lane: (lo, hi)
      reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh][tig])[wq] = sh;
      reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh][tig])[wq] = 0u;
      reinterpret_cast<uint32_t*>(&s.qs[0][quarter][2 * hh + 1][tig])[wq] = sl;
      reinterpret_cast<uint32_t*>(&s.qs[1][quarter][2 * hh + 1][tig])[wq] = sh;
      reinterpret_cast<uint32_t*>(&s.qb[0][quarter][2 * hh][tig])[wb] = qh;
      reinterpret_cast<uint32_t*>(&s.qb[0][quarter][2 * hh + 1][tig])[wb] = ql;
    } else {
      reinterpret_cast<uint32_t*>(&s.qs[0][quarter][j][tig])[wq] = sh;
      reinterpret_cast<uint32_t*>(&s.qs[1][quarter][j][tig])[wq] = sl;
      reinterpret_cast<uint32_t*>(&s.qb[0][quarter][j][tig])[wb] = qh;
      reinterpret_cast<uint32_t*>(&s.qb[NB - 1][quarter][j][tig])[wb] = ql;
    }
  }
  fence_proxy_async();  // q staged in stage buffers that bulk copies fill next
}

// The stage buffer mirrors the packed tile from kStageOff on, byte for byte.
template <int BITS>
constexpr bool kStageMirrorsTile =
    offsetof(TileBuf<BITS>, vc) == kOffVc<BITS> - kStageOff && offsetof(TileBuf<BITS>, sk) == kOffSk<BITS> - kStageOff &&
    offsetof(TileBuf<BITS>, sv) == kOffSv<BITS> - kStageOff && offsetof(TileBuf<BITS>, zv) == kOffZv<BITS> - kStageOff &&
    offsetof(TileBuf<BITS>, outl) == kTileBytes<BITS> - kStageOff && kOffKc<BITS> == kStageOff;
static_assert(kStageMirrorsTile<2> && kStageMirrorsTile<3> && kStageMirrorsTile<4> && kStageMirrorsTile<8>,
              "stage layout");

// The packed tiles of one (batch, kv-head) unit: tile 0, the tile stride, and
// the bytes a stage takes (from kStageOff to the tile's end).
struct UnitSrc {
  const uint8_t* tiles;
  uint32_t stride;
  uint32_t copy;
};

template <int BITS>
__device__ __forceinline__ UnitSrc unit_src(const CacheView& cv, long unit) {
  return UnitSrc{tile_at<BITS>(cv, unit, 0), (uint32_t)cv.tile_bytes, (uint32_t)(cv.tile_bytes - kStageOff)};
}

// One bulk copy of packed tile `tile` into a stage (one lane).
template <int BITS>
__device__ __forceinline__ void issue_tile(TileBuf<BITS>& tb, unsigned long long* bar, const UnitSrc& u,
                                           int tile) {
  mbar_expect_tx(bar, u.copy);
  bulk_g2s(&tb, u.tiles + (long)tile * u.stride + kStageOff, u.copy, bar);
}

// beta = zK x q of the key group of each tile does not depend on the token,
// so it is taken apart from the scores, for sixteen tiles of a warp per MMA:
// rows g and g + 8 of the A operand are the key zeros of tiles k0 + g and
// k0 + g + 8 of the warp, read from global memory (the stages do not hold
// them), k runs over the channels of a quarter, and B is the q table of the
// quarter (q hi / lo, the words of zero-point words 0 and 2, then 1 and 3).
// Lane (g, tig) loads, of the zero vector (channel-pair order, see
// pair_words), the 16-byte chunk zk_chunk(tig, quarter): the words Z0..Z3
// that its A fragments take.  Rows past the warp's last tile load zeros.
template <int BITS>
__device__ __forceinline__ int zk_chunk(int tig, int q) {
  // pair_words: block q >> 1, words 4 (q & 1) .. + 3 of pair block tig + 4
  // (q >> 1) at 2 and 3 bits; block q, pair block tig + 4 q at 4 bits; the
  // four words from 16 tig + 4 q at 8 bits
  return BITS <= 3 ? 2 * tig + 8 * (q >> 1) + (q & 1) : (BITS == 4 ? tig + 4 * q : 4 * tig + q);
}

template <int BITS>
__device__ __forceinline__ void load_zk(const UnitSrc& us, int t_first, int n_mine, int k0, int g, int tig,
                                        uint4 (&z)[2][4]) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int k = k0 + g + 8 * r;
    const uint4* v = reinterpret_cast<const uint4*>(us.tiles + (long)(t_first + kWarps * k) * us.stride + kOffZk);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      z[r][q] = k < n_mine ? __ldg(v + zk_chunk<BITS>(tig, q)) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The MMAs of one sixteen-tile block: D[row][column] accumulates beta of the
// row's tile for the table's column (one key block: (head, hi / lo); two:
// head, one table per part), summed over the parts into the warp's beta rows
// (k0 mod kBetaTiles) + g and + g + 8.
template <int NB>
__device__ __forceinline__ void beta_mma(const PackedState<NB>& ws, const uint4 (&z)[2][4], int g, int tig,
                                         float* rows) {
  float D[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) D[nb][i] = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const uint4 qb = ws.qb[nb][q][g][tig];
      mma16816(D[nb], z[0][q].x, z[1][q].x, z[0][q].z, z[1][q].z, qb.x, qb.y);
      mma16816(D[nb], z[0][q].y, z[1][q].y, z[0][q].w, z[1][q].w, qb.z, qb.w);
    }
  if constexpr (NB == 1) {
    rows[g * 4 + tig] = D[0][0] + D[0][1];
    rows[(g + 8) * 4 + tig] = D[0][2] + D[0][3];
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rows[g * 8 + 2 * tig + i] = D[0][i] + D[NB - 1][i];
      rows[(g + 8) * 8 + 2 * tig + i] = D[0][2 + i] + D[NB - 1][2 + i];
    }
  }
}

// The same from a source address, issued by the lanes where `p` holds (one
// lane) with predicated instructions, so that the warp does not diverge;
// the proxy fence orders the warp's earlier reads of the stage before the
// copy's writes.
template <int BITS>
__device__ __forceinline__ void issue_tile_if(bool p, TileBuf<BITS>& tb, unsigned long long* bar,
                                              const uint8_t* src, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p fence.proxy.async.shared::cta;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %4;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%1], [%2], %4, [%3];\n\t}"
      ::"r"((int)p), "r"(smem_u32(&tb)), "l"(src), "r"(smem_u32(bar)), "r"(bytes)
      : "memory");
}

// Packed tiles [tile0, tile1) of one (batch, kv-head, head chunk) on the
// tensor cores.  Warp w takes tiles tile0 + w, + kWarps, ... through its own
// ring of staged tiles (lane 0 issues the copies; no CTA barrier in the
// loop).  Leaves each warp's (max, sum) per head in s_m / s_l and its output
// in its merge area.
template <int BITS, int NB>
__device__ void packed_split(const CacheView& cv, const AttnArgs& a, const SmemView<BITS, NB>& sv, long unit, int b,
                             int j0, int nh, int tile0, int tile1, float (&s_m)[kWarps][kNH],
                             float (&s_l)[kWarps][kNH]) {
  const int kStages = sv.S;
  PackedState<NB>& ws = sv.ps();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int n_mine = tile0 + warp < tile1 ? (tile1 - tile0 - warp + kWarps - 1) / kWarps : 0;
  unsigned char* const ring = reinterpret_cast<unsigned char*>(sv.ring(warp));
  auto st = [&](int k) -> TileBuf<BITS>& { return *reinterpret_cast<TileBuf<BITS>*>(ring + (size_t)k * sv.stride); };
  unsigned long long* bars = ws.bar[warp];
  const float* const qo = sv.qo();  // q for the outlier channels (when the cache keeps them)
  float qv8[8];
  load_q8(a, b, j0, nh, qv8);

  if (lane == 0) {
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
  if (!wait_first && lane == 0 && issued > 0) issue_tile<BITS>(st(0), &bars[0], us, t_first);
  // the key zeros of the first sixteen tiles are loaded before the tables
  // are built (unless the tiles may still be written by the kernel before)
  uint4 z[2][4];
  if (!wait_first) load_zk<BITS>(us, t_first, n_mine, 0, g, tig, z);
  build_q_tables<BITS, NB>(sv, a, qv8, cv.n_out > 0);
  __syncthreads();
  if (wait_first) grid_dependency_wait();
  if (lane == 0)
    for (int k = wait_first ? 0 : 1; k < issued; ++k) issue_tile<BITS>(st(k), &bars[k], us, t_first + kWarps * k);
  float* const brows = &ws.beta[warp][0][0];
  if (n_mine > 0) {
    if (wait_first) load_zk<BITS>(us, t_first, n_mine, 0, g, tig, z);
    beta_mma<NB>(ws, z, g, tig, brows);
    if (n_mine > 16) {
      load_zk<BITS>(us, t_first, n_mine, 16, g, tig, z);
      beta_mma<NB>(ws, z, g, tig, brows + 16 * 4 * NB);
    }
    __syncwarp();
  }
  float ks[NB], m_run[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    ks[nb] = ws.qscale[NB == 1 ? tig : 2 * tig + nb];
    m_run[nb] = -INFINITY;
  }

  float O[8][4], Z[4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) O[mt][i] = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) Z[i] = 0.0f;

  // Tile k's scores are computed one iteration ahead of its values: the
  // scores of tile k + 1 and the values of tile k form one straight-line
  // block (the wait for tile k + 1 comes first), so that their independent
  // MMA chains can interleave.  One loop body walks the ring with the stage
  // as a run-time index.
  int done = 0;
  bool failed = false;
  uint32_t pb[2][2];  // the staged tile's weights as value B fragments
  if (n_mine > 0) {
    bool ok = mbar_try_wait(&bars[0], 0u);
    if (!ok) ok = mbar_wait(&bars[0], 0u);
    if (__any_sync(kFull, !ok)) {
      failed = true;
    } else {
      float sc[NB][4], mb[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mb[nb] = 0.0f;
      key_scores<BITS, NB>(ws, st(0), g, tig, ks, mb, cv.n_out, qo, brows, sc);
      softmax_p<NB>(sc, g, tig, m_run, O, Z, pb);
    }
  }
  int k = 0, sk = 0;     // tile whose values are next, and its stage
  uint32_t parn = 0;     // phase parity of the stage of tile k + 1
  // source of the next tile to stage (tile k + kStages of this warp)
  const long src_step = (long)kWarps * us.stride;
  const uint8_t* next_src = us.tiles + (long)(t_first + kWarps * kStages) * us.stride + kStageOff;
  while (!failed && k + 1 < n_mine) {
    const int sn = sk + 1 == kStages ? 0 : sk + 1;  // stage of tile k + 1
    if (sn == 0) parn ^= 1u;
    if (!__all_sync(kFull, mbar_try_wait(&bars[sn], parn))) {
      const bool ok = mbar_wait(&bars[sn], parn);
      if (__any_sync(kFull, !ok)) {
        failed = true;
        break;
      }
    }
    const int kb = (k + 1) % kBetaTiles;  // beta row of tile k + 1
    if (kb == 0) {
      // the next block of kBetaTiles tiles (every row of the last one is read)
      __syncwarp();
      uint4 zz[2][4];
      load_zk<BITS>(us, t_first, n_mine, k + 1, g, tig, zz);
      beta_mma<NB>(ws, zz, g, tig, brows);
      if (k + 17 < n_mine) {
        load_zk<BITS>(us, t_first, n_mine, k + 17, g, tig, zz);
        beta_mma<NB>(ws, zz, g, tig, brows + 16 * 4 * NB);
      }
      __syncwarp();
    }
    float sc[NB][4];
    key_scores<BITS, NB>(ws, st(sn), g, tig, ks, m_run, cv.n_out, qo, brows + kb * 4 * NB, sc);
    value_acc<BITS>(st(sk), pb, g, tig, O, Z);
    done = k + 1;
    __syncwarp();  // every lane is done with stage sk
    const bool more = k + kStages < n_mine;
    issue_tile_if<BITS>(more && lane == 0, st(sk), &bars[sk], next_src, us.copy);
    next_src += src_step;
    issued += more;
    softmax_p<NB>(sc, g, tig, m_run, O, Z, pb);
    ++k;
    sk = sn;
  }
  if (!failed && n_mine > 0) {
    value_acc<BITS>(st(sk), pb, g, tig, O, Z);  // the last tile's values
    done = n_mine;
  }
  if (done < n_mine) {
    // A wait timed out: record it, and let every copy still in flight land
    // before the warp's buffers are reused (each wait bounded again).
    if (lane == 0) atomicOr(a.status, 1);
    for (int kk = done; kk < issued; ++kk) mbar_wait(&bars[kk % kStages], (uint32_t)((kk / kStages) & 1));
    __syncwarp();
  } else if (lane == 0) {
    // every copy has landed: the barriers' memory may be reused
    for (int kk = 0; kk < kStages; ++kk) mbar_inval(&bars[kk]);
  }

  // ---- this warp's partial: max, sum and output per head ----
  // The value columns of lane (g, tig) are heads 2 tig and 2 tig + 1: their
  // weight sums are Z[2], Z[3] (the all-ones rows); the running max of head
  // hd(nb) of key_scores is m_run[nb] of the lanes with this tig.
  if (g == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if constexpr (NB == 2) s_m[warp][2 * tig + i] = n_mine > 0 ? m_run[i] : -INFINITY;
      else s_m[warp][4 * i + tig] = i == 0 && n_mine > 0 ? m_run[0] : -INFINITY;
    }
    s_l[warp][2 * tig] = Z[2];
    s_l[warp][2 * tig + 1] = Z[3];
  }
  // z-term of value group gp for heads (2 tig, 2 tig + 1): Z[0], Z[1] of lane (gp, tig)
  float zt[4][2];
#pragma unroll
  for (int gp = 0; gp < 4; ++gp) {
    zt[gp][0] = __shfl_sync(kFull, Z[0], 4 * gp + tig);
    zt[gp][1] = __shfl_sync(kFull, Z[1], 4 * gp + tig);
  }
  if (n_mine == 0) return;  // no tile: the area stays unwritten (max -inf)
  float* oa = sv.merge_area(warp, kPathMma) + (2 * tig) * kHeadDim;
  float* ob = oa + kHeadDim;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int gp = mt >> 1, hm = mt & 1;
    // code positions of rows g and g + 8 of m-tile mt
    const int i_lo = BITS <= 3 ? 4 * (gp & 1) + 2 * hm : 2 * hm;
    const int ch = 32 * gp + 4 * g + 2 * hm;
    const float f_lo = kTwo24 * code_scale<BITS>(i_lo);
    const float f_hi = kTwo24 * code_scale<BITS>(i_lo + 1);
    oa[ch] = O[mt][0] * f_lo + zt[gp][0];
    ob[ch] = O[mt][1] * f_lo + zt[gp][1];
    oa[ch + 1] = O[mt][2] * f_hi + zt[gp][0];
    ob[ch + 1] = O[mt][3] * f_hi + zt[gp][1];
  }
}

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

// Merge n <= kMergeGroup partials [n][kNH][D] (outputs) and [n][kNH][2]
// (max, sum) of head j: lane l takes channels 4l..4l+3; every load is issued
// before the first is used.  Returns the merged (unnormalized) output quad,
// max and sum of head j.
__device__ __forceinline__ void merge_partials(const float* po, const float* pml, int n, int j, float4& o4,
                                               float& m_out, float& l_out) {
  const int lane = threadIdx.x & 31;
  float4 v[kMergeGroup];
#pragma unroll
  for (int k = 0; k < kMergeGroup; ++k)
    v[k] = k < n ? __ldcg(reinterpret_cast<const float4*>(po + ((long)k * kNH + j) * kHeadDim) + lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  const float2 ml = lane < n ? __ldcg(reinterpret_cast<const float2*>(pml + ((long)lane * kNH + j) * 2))
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
template <int BITS, int NB>
__device__ void fused_tail(const CacheView& cv, const AttnArgs& a, const SeqPlan p, const SmemView<BITS, NB>& sv,
                           long unit, int b, int j0, int nh, float (&s_m)[kWarps][kNH],
                           float (&s_l)[kWarps][kNH]) {
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
        ot += e * sv.merge_area(w, kPathMma)[j * kHeadDim + d];
      }
    }
    pm[j] = M;
    pl[j] = lt;
    po[j] = ot;
  }
  __syncthreads();  // the warps' slots are read; the tail may overwrite them
  float* mo0 = sv.merge_area(0, kPathTail);
  uint32_t round = 0;
  for (int c0 = p.t_tail; c0 < p.l; c0 += kTailTok, ++round) {
    tail_split<BITS, NB>(cv, a, p, sv.tail(), mo0, unit, b, j0, nh, c0, round, s_m, s_l);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
      const float tm = s_m[0][j];
      const float M = fmaxf(pm[j], tm);
      const float e1 = pm[j] == -INFINITY ? 0.0f : fast_exp2(pm[j] - M);
      const float e2 = tm == -INFINITY ? 0.0f : fast_exp2(tm - M);
      // (rows of heads the tail does not serve are not written: max -inf)
      po[j] = po[j] * e1 + (tm == -INFINITY ? 0.0f : mo0[j * kHeadDim + d] * e2);
      pl[j] = pl[j] * e1 + s_l[0][j] * e2;
      pm[j] = M;
    }
    __syncthreads();  // before the next round overwrites the staged rows
  }
  float* out0 = sv.merge_area(0, kPathMma);
#pragma unroll
  for (int j = 0; j < kNH; ++j) out0[j * kHeadDim + d] = po[j];
  if (d < kWarps * kNH) {
    const int w = d / kNH, j = d % kNH;
    float mj = pm[0], lj = pl[0];
#pragma unroll
    for (int i = 1; i < kNH; ++i) {
      mj = j == i ? pm[i] : mj;
      lj = j == i ? pl[i] : lj;
    }
    s_m[w][j] = w == 0 ? mj : -INFINITY;
    s_l[w][j] = w == 0 ? lj : 0.0f;
  }
  __syncthreads();
}

// grid (splits, H * head_chunks, B), 128 threads.
template <int BITS, int NB>
__global__ void __launch_bounds__(128, attn_ctas_per_sm(BITS, NB))
    attn_kernel(CacheView cv, AttnArgs a, const SeqLens lens) {
  extern __shared__ __align__(16) unsigned char smem_raw[];  // attn_stages: the tail or the packed layout
  const SmemView<BITS, NB> sv{smem_raw, a.stages, (uint32_t)(cv.tile_bytes - kStageOff)};
  __shared__ float s_m[kWarps][kNH], s_l[kWarps][kNH];
  __shared__ bool s_last;

  // Programmatic dependents of this launch (an overlapping attention call,
  // the next decode step's append) may start early.  An ordinary or an
  // overlapping launch lets them start at once: it writes nothing they read
  // (its workspace and out aside, which they wait for before writing), and
  // every kernel before it has completed or writes nothing it reads.  A
  // decode step's attention lets them start only once its append has
  // completed (before the merge below), so that no early start ever runs
  // ahead of a cache write.
  const bool step_launch = a.pdl == kPdlAll || a.pdl == kPdlTail;
  const int s = blockIdx.x;
  const int nhc = gridDim.y / cv.H;
  const int h = nhc == 1 ? (int)blockIdx.y : (int)blockIdx.y / nhc;
  const int hc = nhc == 1 ? 0 : (int)blockIdx.y % nhc;
  const int b = blockIdx.z;
  const long gid = (long)b * gridDim.y + blockIdx.y;  // (batch, kv-head, head chunk)
  // An overlapping launch releases its dependents at once, once its
  // generation ticket is taken (take_ticket); a decode step's attention
  // releases them once its append has completed (before the merge below),
  // an ordinary launch at its exit.
  const bool tickets = a.epoch_on && a.pdl != 0;
  unsigned gen = 0;  // thread 0: this launch's generation for the group
  if (tickets && threadIdx.x == 0) gen = take_ticket(a, gid);
  if (a.pdl == kPdlOverlap) {
    if (threadIdx.x == 0) gen = ticket_gen(gen);
    __syncthreads();
    grid_launch_dependents();
  }
  const int grp = a.Hq / cv.H;
  const int j0 = h * grp + hc * kNH;
  const int nh = min(kNH, grp - hc * kNH);
  const long unit = (long)b * cv.H + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  (void)gid;
  // this sequence's plan; splits past its own count have nothing to do (and
  // are not counted by its merge)
  const SeqPlan p = lens.uniform >= 0 ? a.plan : make_plan(lens.l[b], cv.R, cv.policy, a.scfg);
  if (s >= p.splits) {
    if (step_launch && threadIdx.x == 0) gen = ticket_gen(gen);  // the ticket is in before the exit
    return;
  }
  const int path = s < p.tail_splits ? kPathTail : kPathMma;

  if (path == kPathTail) {
    // the tail reads the rings the append writes
    if (a.pdl == kPdlAll || a.pdl == kPdlTail) grid_dependency_wait();
    tail_split<BITS, NB>(cv, a, p, sv.tail(), sv.merge_area(0, kPathTail), unit, b, j0, nh,
                         p.t_tail + s * kTailTok, 0u, s_m, s_l);
  } else {
    // ---- tensor cores: packed tiles [sp*chunk, min(t_tail, (sp+1)*chunk)) ----
    const int sp = s - p.tail_splits;
    const int tile0 = sp * p.chunk / 32;
    const int tile1 = min(p.t_tail, (sp + 1) * p.chunk) / 32;
    packed_split<BITS, NB>(cv, a, sv, unit, b, j0, nh, tile0, tile1, s_m, s_l);
  }
  __syncthreads();
  if (path == kPathMma && p.tail_fused && s == p.splits - 1) {
    if (a.pdl == kPdlTail) grid_dependency_wait();  // the tail reads what the append wrote
    fused_tail<BITS, NB>(cv, a, p, sv, unit, b, j0, nh, s_m, s_l);
  }
  // a decode step's attention releases its dependents once its append has
  // completed
  if (step_launch) {
    grid_dependency_wait();
    if (threadIdx.x == 0) gen = ticket_gen(gen);
    __syncthreads();
    grid_launch_dependents();
  }
  // an overlapping launch orders its first workspace write of the group after
  // the previous call on this workspace has finished with the group's slots
  // (see epoch_wait); a wait that gives up sets bit 2 of the status word
  if (a.pdl == kPdlOverlap && a.epoch_on) {
    if (threadIdx.x == 0 && !epoch_wait(a.epochs + 2 * gid + 1, gen)) atomicOr(a.status, 2);
    __syncthreads();
  }

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
        if (s_m[w][j] == -INFINITY) continue;  // an empty warp (its area is not written)
        const float e = fast_exp2(s_m[w][j] - M);
        lt += e * s_l[w][j];
        ot += e * sv.merge_area(w, path)[j * kHeadDim + d];
      }
    }
    const long pidx = (gid * a.scfg.max_splits + s) * kNH + j;
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
  // warp w merges heads w and w + kWarps
  float4 o4[2];
  float lsum_h[2], m_h[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = warp + kWarps * hh;
    if (j < nh)
      merge_partials(a.ws_o + (gid * a.scfg.max_splits + g_lo) * kNH * kHeadDim, a.ws_ml + (gid * a.scfg.max_splits + g_lo) * kNH * 2,
                     g_n, j, o4[hh], m_h[hh], lsum_h[hh]);
  }
  if (n_grp > 1) {
    // a group result: write it, then count the group in
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int j = warp + kWarps * hh;
      if (j < nh) {
        const long pidx = (gid * a.merge_groups + grp_i) * kNH + j;
        *reinterpret_cast<float4*>(a.ws_o1 + pidx * kHeadDim + 4 * lane) = o4[hh];
        if (lane == 0) {
          a.ws_ml1[pidx * 2] = m_h[hh];
          a.ws_ml1[pidx * 2 + 1] = lsum_h[hh];
        }
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
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int j = warp + kWarps * hh;
      if (j < nh)
        merge_partials(a.ws_o1 + gid * a.merge_groups * kNH * kHeadDim, a.ws_ml1 + gid * a.merge_groups * kNH * 2,
                       n_grp, j, o4[hh], m_h[hh], lsum_h[hh]);
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = warp + kWarps * hh;
    if (j >= nh) continue;
    const float inv = 1.0f / lsum_h[hh];
    const float r[4] = {o4[hh].x * inv, o4[hh].y * inv, o4[hh].z * inv, o4[hh].w * inv};
    const long oi = ((long)b * a.Hq + j0 + j) * kHeadDim + 4 * lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (a.q_dtype == kF32) static_cast<float*>(a.out)[oi + i] = r[i];
      else if (a.q_dtype == kF16) static_cast<__half*>(a.out)[oi + i] = __float2half_rn(r[i]);
      else static_cast<__nv_bfloat16*>(a.out)[oi + i] = __float2bfloat16_rn(r[i]);
    }
  }
  // the group's slots are free for the next call on this workspace: every
  // thread's reads of them precede the barrier, the release orders them
  if (tickets) {
    __syncthreads();
    if (threadIdx.x == 0) st_release_u32(a.epochs + 2 * gid + 1, (gen + 1u) & kGenMask);
  }
  // An overlapping launch completes only after the launch before it: group
  // 0's final CTA waits for it last of all, so that whatever follows this
  // launch on the stream (a copy, a memset, a host read after a sync) also
  // follows every launch before it; the other CTAs exit at once.
  if (a.pdl == kPdlOverlap && gid == 0) grid_dependency_wait();
}

}  // namespace

// Stages per warp for a tile of `stride` bytes: as many as attn_ctas_per_sm
// CTAs per SM leave room for (228 KB of shared memory per SM; per CTA 1 KB
// reserved by the system and the kernel's static arrays), at least two and
// at most kMaxStages; *smem is the dynamic size (the packed layout, with
// the copy of q when the cache keeps n_out > 0 outlier channels, or the tail
// split's if larger).
template <int BITS, int NB>
int attn_stages(uint32_t stride, int n_out, size_t* smem) {
  const size_t per_cta = (size_t)228 * 1024 / attn_ctas_per_sm(BITS, NB) - 1024 - 512;
  const size_t q_copy = n_out > 0 ? (size_t)kNH * kHeadDim * 4 : 0;
  const size_t fixed = sizeof(PackedState<NB>) + q_copy + 16;
  int S = (int)((per_cta - fixed) / ((size_t)kWarps * stride));
  S = S < 2 ? 2 : (S > kMaxStages ? kMaxStages : S);
  const size_t packed = packed_state_off(S, stride) + sizeof(PackedState<NB>) + q_copy;
  *smem = packed > sizeof(TailSmem<BITS>) ? packed : sizeof(TailSmem<BITS>);
  return S;
}

template <int BITS, int NB>
constexpr bool kTailFits =
    attn_ctas_per_sm(BITS, NB) * (sizeof(TailSmem<BITS>) + 1024 + 512) <= 228 * 1024;
static_assert(kTailFits<2, 1> && kTailFits<2, 2> && kTailFits<3, 1> && kTailFits<3, 2> && kTailFits<4, 1> &&
                  kTailFits<4, 2> && kTailFits<8, 1> && kTailFits<8, 2>,
              "the tail split's layout fits the CTAs of an SM");

template <int BITS, int NB>
cudaError_t launch_bits(const dim3& grid, const CacheView& cv, AttnArgs a, const SeqLens& lens,
                        cudaStream_t st) {
  size_t smem = 0, cap = 0;
  a.stages = attn_stages<BITS, NB>((uint32_t)(cv.tile_bytes - kStageOff), cv.n_out, &smem);
  // The shared-memory opt-in is a per-device function attribute: set to the
  // largest size any outlier count asks for (the same on every call, so
  // that calls from several host threads cannot shrink it under another's
  // launch); setting it costs a host call only.
  const uint32_t plain = (uint32_t)(cv.tile_bytes - kStageOff - outlier_block_bytes(cv.n_out));
  for (int n = 0; n <= kMaxOutliers; ++n) {
    size_t sz = 0;
    attn_stages<BITS, NB>(plain + (uint32_t)outlier_block_bytes(n), n, &sz);
    cap = sz > cap ? sz : cap;
  }
  const cudaError_t e =
      cudaFuncSetAttribute(attn_kernel<BITS, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cap);
  if (e != cudaSuccess) return e;
  if (!a.pdl) {
    attn_kernel<BITS, NB><<<grid, 128, smem, st>>>(cv, a, lens);
    return cudaGetLastError();
  }
  // a programmatic dependent of the kernel before it on the stream
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(128);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, attn_kernel<BITS, NB>, cv, a, lens);
}

cudaError_t launch_wait_probe(int* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

template <int NB>
cudaError_t launch_nb(const dim3& grid, const CacheView& cv, const AttnArgs& a, const SeqLens& lens,
                      cudaStream_t st) {
  switch (cv.bits) {
    case 2: return launch_bits<2, NB>(grid, cv, a, lens, st);
    case 3: return launch_bits<3, NB>(grid, cv, a, lens, st);
    case 4: return launch_bits<4, NB>(grid, cv, a, lens, st);
    default: return launch_bits<8, NB>(grid, cv, a, lens, st);
  }
}

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a, const SeqLens& lens, cudaStream_t st) {
  const int grp = a.Hq / cv.H;
  const int nhc = (grp + kNH - 1) / kNH;
  const dim3 grid(a.splits, cv.H * nhc, cv.B);
  return attn_key_blocks(grp) == 2 ? launch_nb<2>(grid, cv, a, lens, st) : launch_nb<1>(grid, cv, a, lens, st);
}

}  // namespace kivi
