// kivi_internal.cuh -- shared definitions of the CUDA library (internal).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

constexpr int kHeadDim = 128;  // D supported by the kernels
constexpr int kGroup = 32;     // G supported by the kernels
constexpr int kTargetSMs = 152;    // GB300 SM count used by the split policy
constexpr int kAttnCtasPerSm = 4;  // attention CTAs resident per SM (registers, shared memory)
constexpr int kHeadChunk = 4;      // query heads per attention CTA
constexpr int kMergeGroup = 16;    // split partials merged by one CTA (two levels at most)
constexpr int kTailTok = 64;       // tail tokens per tail split
constexpr int kMaxSplits = kMergeGroup * kMergeGroup;

// Device view of one cache: the packed tile store, the two rings and the shape.
struct CacheView {
  uint8_t* tiles;  // [B][H][Tcap / kGroup] tiles of kTileBytes<bits>
  __half* ring_k;
  __half* ring_v;
  int B, H, R, Tcap, bits;
  int W;  // ring slots: token t of a unit is in slot t mod W
};

// A packed tile holds everything quantized about tokens [32j, 32j + 32) of a
// unit, so that one bulk copy stages it:
//   [0, 32 RB)                key code rows (RB = D * bits / 8 bytes each)
//   [32 RB, 64 RB)            value code rows (group-interleaved)
//   kOffSk: scale[D] (f16)    of the tile's key group, one per channel
//   kOffZk: zero[D]
//   kOffSv: scale[32][D / G]  value groups, per token
//   kOffZv: zero[32][D / G]
template <int BITS>
constexpr int kRowBytes = kHeadDim * BITS / 8;
template <int BITS>
constexpr int kOffVc = kGroup * kRowBytes<BITS>;
template <int BITS>
constexpr int kOffSk = 2 * kGroup * kRowBytes<BITS>;
template <int BITS>
constexpr int kOffZk = kOffSk<BITS> + 2 * kHeadDim;
template <int BITS>
constexpr int kOffSv = kOffSk<BITS> + 4 * kHeadDim;
template <int BITS>
constexpr int kOffZv = kOffSk<BITS> + 6 * kHeadDim;
template <int BITS>
constexpr int kTileBytes = kOffSk<BITS> + 8 * kHeadDim;
static_assert(kTileBytes<2> == 3072 && kTileBytes<4> == 5120, "tile sizes");
static_assert(kGroup * (kHeadDim / kGroup) * 2 == 2 * kHeadDim, "value scale block size");

// Key scales / zeros of a tile are stored in channel-pair order: 32-bit word
// i of pair block m holds the fp16 pair (channel P m + i, channel P m + i +
// P / 2), P = 16 at 2 bits and 8 at 4 bits -- the two values one B-fragment
// register of the score product takes.  kscale_pos(c) is channel c's fp16
// slot.
template <int BITS>
__host__ __device__ constexpr int kscale_pos(int c) {
  constexpr int P = BITS == 2 ? 16 : 8;
  return P * (c / P) + 2 * (c % (P / 2)) + (c % P) / (P / 2);
}

// Value scales / zeros of a tile are stored by token pair: with t = 8a + 4h +
// r (r < 4), 32-bit word 4 (4a + r) + gp holds group gp of tokens (8a + r,
// 8a + r + 4), the pair that one B-fragment register of the value product
// takes.  vscale_pos(t, gp) is the fp16 slot of token t, group gp.
__host__ __device__ constexpr int vscale_pos(int t, int gp) {
  return 32 * (t / 8) + 8 * (t % 4) + 2 * gp + (t / 4) % 2;
}

// Tile `tile` (tokens [32 tile, 32 tile + 32)) of unit `unit`.
template <int BITS>
__host__ __device__ __forceinline__ uint8_t* tile_at(const CacheView& cv, long unit, long tile) {
  return cv.tiles + (unit * (cv.Tcap / kGroup) + tile) * (long)kTileBytes<BITS>;
}

// Input dtype codes (same values as kivi_dtype).
enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

cudaError_t launch_quantize_prefill(const CacheView& cv, const void* k,
                                    const void* v, int dtype, int T, int nq_k,
                                    int nq_v, cudaStream_t st);

cudaError_t launch_append(const CacheView& cv, const void* k, const void* v,
                          int dtype, int t, cudaStream_t st);

// n tokens appended to a cache of length l0 (k, v: [B][H][n][D] of dtype):
// key groups [nq_k0, nq_k1) and value tokens [nq_v0, nq_v1) become
// quantized, then the last min(n, R) tokens go to the ring.
cudaError_t launch_append_tokens(const CacheView& cv, const void* k, const void* v, int dtype,
                                 int l0, int n, int nq_k0, int nq_k1, int nq_v0, int nq_v1,
                                 cudaStream_t st);

struct AttnArgs {
  const void* q;
  void* out;
  int q_dtype;
  int Hq;
  float scale_log2;  // softmax scale * log2(e)
  int l, nq_k, nq_v;
  // Context split: splits s < tail_splits cover the tail [t_tail, l) (t_tail
  // = nq_v rounded down to 32), kTailTok tokens each from t_tail + s*kTailTok;
  // split tail_splits + i covers the packed tiles [i*chunk, min(t_tail,
  // (i+1)*chunk)).
  // With tail_fused set there are no tail splits: the last packed split also
  // takes the tail, after its tiles (when the one-wave budget leaves no room).
  int t_tail;
  int tail_splits, splits, chunk, tail_fused;
  // Split partials of attention group gid = (b, kv-head, head chunk):
  float* ws_o;        // [gid][splits][kHeadChunk][D]  output sums
  float* ws_ml;       // [gid][splits][kHeadChunk][2]  (max in log2 units, sum)
  float* ws_o1;       // [gid][merge_groups][kHeadChunk][D]  merged groups of kMergeGroup splits
  float* ws_ml1;      // [gid][merge_groups][kHeadChunk][2]
  int merge_groups;   // stride of the group arrays (ceil(max splits / kMergeGroup))
  int* counters;      // [gid][merge_groups] CTAs finished per split group; 0 between calls
  int* counters2;     // [gid] split groups finished; 0 between calls
  int* status;        // set nonzero when a bounded wait for staged data timed out
};

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a,
                             cudaStream_t st);

}  // namespace kivi
