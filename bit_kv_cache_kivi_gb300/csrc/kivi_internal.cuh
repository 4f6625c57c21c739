// kivi_internal.cuh -- shared definitions of the CUDA library (internal).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

constexpr int kHeadDim = 128;  // D supported by the kernels
constexpr int kGroup = 32;     // G supported by the kernels
constexpr int kTargetSMs = 152;    // GB300 SM count used by the split policy
constexpr int kHeadChunk = 8;      // query heads per attention CTA
// Key blocks of a head chunk: the score product takes four query heads per
// MMA (each as an fp16 hi / lo pair of columns), so chunks of up to four
// heads need one block and chunks of five to eight need two.
__host__ __device__ constexpr int attn_key_blocks(int grp) { return (grp < kHeadChunk ? grp : kHeadChunk) > 4 ? 2 : 1; }
// Attention CTAs resident per SM (registers, shared memory): four, except
// that two 9 KB staged tiles per warp at 8 bits leave room for two, and the
// two key blocks' query tables beside two 5 KB stages per warp at 4 bits for
// three.
__host__ __device__ constexpr int attn_ctas_per_sm(int bits, int nb) {
  return bits == 8 ? 2 : (bits == 4 && nb == 2 ? 3 : 4);
}
constexpr int kMergeGroup = 16;    // split partials merged by one CTA (two levels at most)
constexpr int kTailTok = 64;       // tail tokens per tail split
constexpr int kMaxSplits = kMergeGroup * kMergeGroup;

constexpr int kMaxVarBatch = 1024;  // batch limit for per-sequence lengths
constexpr int kMaxOutliers = 4;     // fp16 outlier key channels per key group, at most

// Device view of one cache: the packed tile store, the two rings and the shape.
struct CacheView {
  uint8_t* tiles;  // [B][H][Tcap / kGroup] tiles of tile_bytes
  __half* ring_k;
  __half* ring_v;
  int B, H, R, Tcap, bits;
  int W;           // ring slots: token t of a unit is in slot t mod W
  int policy;      // 0: Algorithm 1 of the chooblog KIVI review; 1: shared window
  int n_out;       // fp16 outlier key channels per key group (0..kMaxOutliers)
  int tile_bytes;  // kTileBytes<bits> + outlier_block_bytes(n_out)
};

// The lengths of the batch's sequences, passed by value to every launch:
// one length for all, or one per sequence (batch <= kMaxVarBatch).
struct SeqLens {
  int uniform;  // >= 0: every sequence has this length; -1: l[b]
  int n;        // tokens the launch appends to each sequence (0 for attention)
  int u_nq[4];  // uniform: nq_k(l), nq_v(l), nq_k(l + n), nq_v(l + n)
  int l[kMaxVarBatch];
};

__host__ __device__ __forceinline__ int seq_len(const SeqLens& s, int b) {
  return s.uniform >= 0 ? s.uniform : s.l[b];
}

// Quantized counts after l tokens.  Policy 0 (chooblog KIVI review §3.2.2,
// Algorithm 1): keys X_K[:l - l mod R], values X_V[:l - R].  Policy 1
// (veloxquant-mlx "KIVI" How it works, items 3-4): both G*floor((l - R)/G).
__host__ __device__ __forceinline__ int policy_nq_k(int l, int R, int policy) {
  if (policy == 1) return l > R ? (l - R) / kGroup * kGroup : 0;
  return l - l % R;
}
__host__ __device__ __forceinline__ int policy_nq_v(int l, int R, int policy) {
  if (policy == 1) return policy_nq_k(l, R, policy);
  return l > R ? l - R : 0;
}

// Quantized counts of sequence b before and after the launch's n tokens:
// nq_k(l), nq_v(l), nq_k(l + n), nq_v(l + n) (precomputed when uniform).
__device__ __forceinline__ void seq_counts(const SeqLens& s, int b, int R, int policy, int (&c)[4]) {
  if (s.uniform >= 0) {
    c[0] = s.u_nq[0], c[1] = s.u_nq[1], c[2] = s.u_nq[2], c[3] = s.u_nq[3];
  } else {
    const int l = s.l[b];
    c[0] = policy_nq_k(l, R, policy), c[1] = policy_nq_v(l, R, policy);
    c[2] = policy_nq_k(l + s.n, R, policy), c[3] = policy_nq_v(l + s.n, R, policy);
  }
}

// Split configuration of a cache (a function of its shape and of whether
// the launch overlaps the one before it): the budget of splits per attention
// unit, the workspace's bound on splits, a caller's override (0 =
// automatic), and the automatic plan's knobs below.
struct SplitCfg {
  int budget, max_splits, override_splits;
  int min_tiles;         // packed tiles per automatic split, at least
  int fuse_single_tail;  // automatic plans ride a one-split tail on the last packed split
  int fused_discount;    // tiles fewer for the packed split that carries a fused tail
};

// How decode attention covers one sequence of length l: tail splits of
// kTailTok tokens from t_tail = 32 floor(nq_v / 32) (CUDA cores), then packed
// splits of `chunk` tokens over the tiles below t_tail (tensor cores).
// Automatic packed splits fill the budget beside the tail splits, with at
// least min_tiles tiles and a multiple of four each (the four warps of a CTA
// get equal shares); an override asks for that many splits in all.  When the
// budget cannot hold a tail split beside one packed split, or the tail is one
// split and fuse_single_tail is set, the tail rides on the last packed split
// (tail_fused, no tail splits).
struct SeqPlan {
  int l, nq_k, nq_v, t_tail, tail_splits, splits, chunk, tail_fused;
};

__host__ __device__ inline SeqPlan make_plan(int l, int R, int policy, const SplitCfg& sc) {
  SeqPlan p;
  p.l = l;
  p.nq_k = policy_nq_k(l, R, policy);
  p.nq_v = policy_nq_v(l, R, policy);
  const int tt = p.nq_v / 32 * 32;
  p.t_tail = tt;
  p.tail_splits = (l - tt + kTailTok - 1) / kTailTok;
  p.tail_fused = 0;
  const int tiles = tt / 32;
  if (tiles == 0) {
    p.splits = p.tail_splits;
    p.chunk = 32;
    return p;
  }
  if (sc.override_splits <= 0 &&
      (sc.budget < p.tail_splits + 1 || (sc.fuse_single_tail && p.tail_splits == 1))) {
    p.tail_fused = 1;
    p.tail_splits = 0;
  }
  int smax = sc.budget - p.tail_splits;
  if (smax > sc.max_splits - p.tail_splits) smax = sc.max_splits - p.tail_splits;
  if (smax < 1) smax = 1;
  int per;  // tiles per packed split
  if (sc.override_splits > 0) {
    int s = sc.override_splits - p.tail_splits;
    if (s > sc.max_splits - p.tail_splits) s = sc.max_splits - p.tail_splits;
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    per = (tiles + s - 1) / s;
  } else {
    per = (tiles + smax - 1) / smax;
    per = (per + 3) / 4 * 4;
    if (per < sc.min_tiles) per = sc.min_tiles;
    if (p.tail_fused && sc.fused_discount > 0) {
      // the last split runs the tail after its tiles: spread fused_discount
      // of its tiles over the others (as long as the split count holds)
      const int n = (tiles + per - 1) / per;
      int per2 = (tiles + sc.fused_discount + n - 1) / n;
      per2 = (per2 + 3) / 4 * 4;
      if (n > 1 && per2 > per && (n - 1) * per2 < tiles) per = per2;
    }
  }
  p.chunk = per * 32;
  p.splits = p.tail_splits + (tt + p.chunk - 1) / p.chunk;  // no empty split
  return p;
}

// A packed tile holds everything quantized about tokens [32j, 32j + 32) of a
// unit:
//   kOffZk: zero[D] (f16)     of the tile's key group, one per channel
//   kOffKc: 32 key code rows  (RB = D * bits / 8 bytes each)
//   kOffVc: 32 value code rows (group-interleaved)
//   kOffSk: scale[D]          of the tile's key group
//   kOffSv: scale[32][D / G]  value groups, per token
//   kOffZv: zero[32][D / G]
//   then the outlier block, if the cache keeps outlier channels.
// The decode attention stages [kStageOff, tile end) with one bulk copy; it
// reads the key zeros apart, for sixteen tiles at a time (load_zk and
// beta_mma in attention.cu), so they lead the tile.
template <int BITS>
constexpr int kRowBytes = kHeadDim * BITS / 8;
constexpr int kOffZk = 0;
constexpr int kStageOff = 2 * kHeadDim;
template <int BITS>
constexpr int kOffKc = kStageOff;
template <int BITS>
constexpr int kOffVc = kOffKc<BITS> + kGroup * kRowBytes<BITS>;
template <int BITS>
constexpr int kOffSk = kOffKc<BITS> + 2 * kGroup * kRowBytes<BITS>;
template <int BITS>
constexpr int kOffSv = kOffSk<BITS> + 2 * kHeadDim;
template <int BITS>
constexpr int kOffZv = kOffSk<BITS> + 4 * kHeadDim;
template <int BITS>
constexpr int kTileBytes = kOffSk<BITS> + 6 * kHeadDim;
static_assert(kTileBytes<2> == 3072 && kTileBytes<3> == 4096 && kTileBytes<4> == 5120 &&
                  kTileBytes<8> == 9216,
              "tile sizes");

// 3-bit code rows (48 bytes) are two planes: bytes [0, 32) hold the low two
// bits of every code exactly as a 2-bit row (keys LSB-first, values
// group-interleaved), bytes [32, 48) the high bits in eight 16-bit units.
// Key unit 2W + h (W = 0..3, h = 0..1) holds channels 16m + 8h + i for m in
// {W, W + 4} (set s = m / 4) and i = 0..7; value unit w holds channels
// 32 gp + 4w + c of the four groups (set s = gp / 2, i = 4 (gp mod 2) + c).
// (s, i) sits at bit hi_bit3(s, i) of its unit.  With this placement the high
// bit of position i of a 2-bit key word lands two bits above that code's low
// bits after the same shift the low bits take (w for i < 4, w >> 8 above),
// from the unit word as is (set 0, i < 4), shifted by one (set 0, i >= 4),
// with its bytes swapped within each half (set 1, i < 4), or both (set 1,
// i >= 4); the value units follow the same rule per group.
__host__ __device__ constexpr int hi_bit3(int s, int i) {
  return s ? (2 * (i & 3) + 2 + (i >> 2) + 8) & 15 : 2 * (i & 3) + 2 + (i >> 2);
}
constexpr int kHiPlane3 = 32;  // byte offset of the high plane in a 3-bit row

// At 8 bits a code row is 128 bytes, so that rows at a multiple of 128 bytes
// would put the same word of every row in the same shared-memory bank.  The
// rows are therefore stored rotated by whole 16-byte chunks: key row r by
// (r & 1) chunks, value row r by 2 (r & 3) chunks -- logical chunk c of the
// row sits at chunk (c + rot) mod 8.  At 2 and 4 bits nothing is rotated.
template <int BITS>
__host__ __device__ __forceinline__ int krow_chunk(int r, int c) {
  return BITS == 8 ? (c + (r & 1)) & 7 : c;
}
template <int BITS>
__host__ __device__ __forceinline__ int vrow_chunk(int r, int c) {
  return BITS == 8 ? (c + 2 * (r & 3)) & 7 : c;
}
// Byte offset of logical byte i of key / value row r (within the row).
template <int BITS>
__host__ __device__ __forceinline__ int krow_byte(int r, int i) {
  return 16 * krow_chunk<BITS>(r, i >> 4) + (i & 15);
}
template <int BITS>
__host__ __device__ __forceinline__ int vrow_byte(int r, int i) {
  return 16 * vrow_chunk<BITS>(r, i >> 4) + (i & 15);
}
static_assert(kGroup * (kHeadDim / kGroup) * 2 == 2 * kHeadDim, "value scale block size");

// Key scales / zeros of a tile are stored in channel-pair order: 32-bit word
// i of pair block m holds the fp16 pair (channel P m + i, channel P m + i +
// P / 2), P = 16 at 2 and 3 bits, 8 at 4 bits and 4 at 8 bits -- the two values one
// B-fragment register of the score product takes.  kscale_pos(c) is channel
// c's fp16 slot.
template <int BITS>
__host__ __device__ constexpr int kscale_pos(int c) {
  constexpr int P = BITS <= 3 ? 16 : (BITS == 4 ? 8 : 4);
  return P * (c / P) + 2 * (c % (P / 2)) + (c % P) / (P / 2);
}

// Value scales / zeros of a tile are stored by token pair: with t = 8a + 4h +
// r (r < 4), 32-bit word 4 (4a + r) + gp holds group gp of tokens (8a + r,
// 8a + r + 4), the pair that one B-fragment register of the value product
// takes.  vscale_pos(t, gp) is the fp16 slot of token t, group gp.
__host__ __device__ constexpr int vscale_pos(int t, int gp) {
  return 32 * (t / 8) + 8 * (t % 4) + 2 * gp + (t / 4) % 2;
}

// Outlier-aware keys (the "KIVI - 2-bit KV cache quantisation" notebook,
// Exercises item 2): with n_out > 0 a tile ends with an outlier block --
// 16 bytes of channel indices (n_out used, largest max |k| first), then
// vals[32 tokens][n_out] fp16 -- and those channels' codes, scales and zeros
// in the tile are 0.
__host__ __device__ constexpr int outlier_block_bytes(int n_out) { return n_out > 0 ? 16 + 64 * n_out : 0; }

// Tile `tile` (tokens [32 tile, 32 tile + 32)) of unit `unit`.
template <int BITS>
__host__ __device__ __forceinline__ uint8_t* tile_at(const CacheView& cv, long unit, long tile) {
  return cv.tiles + (unit * (cv.Tcap / kGroup) + tile) * (long)cv.tile_bytes;
}

// Input dtype codes (same values as kivi_dtype).
enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// Prefill of an empty cache: sequence b takes the first lens(b) of the
// t_in rows of k, v ([B][H][t_in][D] of dtype).
cudaError_t launch_quantize_prefill(const CacheView& cv, const void* k, const void* v, int dtype,
                                    int t_in, const SeqLens& lens, cudaStream_t st);

// One token appended to every sequence (Algorithm 1 policy), at position
// lens(b) of sequence b.
// trig: let a programmatic dependent (a decode step's attention) start at
// once; 0: no dependent launch starts before the append completes.
cudaError_t launch_append(const CacheView& cv, const void* k, const void* v,
                          int dtype, const SeqLens& lens, cudaStream_t st, int trig = 0);

// n tokens appended to every sequence (k, v: [B][H][n][D] of dtype), to a
// sequence of length l0 = lens(b): its key groups [nq_k(l0), nq_k(l0 + n))
// and value tokens [nq_v(l0), nq_v(l0 + n)) become quantized, then its last
// min(n, W) tokens go to the ring.  trig: the ring kernel lets a dependent
// launch (a decode step's attention) start at once; 0: none starts before
// it completes.
cudaError_t launch_append_tokens(const CacheView& cv, const void* k, const void* v, int dtype,
                                 int n, const SeqLens& lens, cudaStream_t st, int trig = 0);

struct AttnArgs {
  const void* q;
  void* out;
  int q_dtype;
  int Hq;
  float scale_log2;  // softmax scale * log2(e)
  // Context split of a sequence (SeqPlan): splits s < tail_splits cover the
  // tail [t_tail, l), kTailTok tokens each from t_tail + s*kTailTok; split
  // tail_splits + i covers the packed tiles [i*chunk, min(t_tail,
  // (i+1)*chunk)).  With tail_fused set there are no tail splits: the last
  // packed split also takes the tail, after its tiles.
  SeqPlan plan;   // of every sequence when the lengths are uniform
  SplitCfg scfg;  // to plan each sequence on the device otherwise
  int splits;     // grid width: the most splits of any sequence
  // Split partials of attention group gid = (b, kv-head, head chunk):
  // per-split partials, [gid][scfg.max_splits][...]: a fixed stride per group,
  // so that calls with different split counts on one workspace use the same
  // slots for the same group (overlapping calls are ordered per group)
  float* ws_o;        // [gid][max splits][kHeadChunk][D]  output sums
  float* ws_ml;       // [gid][max splits][kHeadChunk][2]  (max in log2 units, sum)
  float* ws_o1;       // [gid][merge_groups][kHeadChunk][D]  merged groups of kMergeGroup splits
  float* ws_ml1;      // [gid][merge_groups][kHeadChunk][2]
  int merge_groups;   // stride of the group arrays (ceil(max splits / kMergeGroup))
  int* counters;      // [gid][merge_groups] CTAs finished per split group; 0 between calls
  int* counters2;     // [gid] split groups finished; 0 between calls
  int* status;        // bit 1: a bounded wait for staged data timed out; bit 2: an epoch wait did
  // [gid][2]: tickets taken by the calls' CTAs (kMaxSplits per call), and the
  // generation up to which calls have finished with the group's slots (both
  // 0 after the workspace was zeroed); epoch_on = 0: none of it (a scratch
  // area zeroed for each call)
  unsigned* epochs;
  int epoch_on;
  int stages;         // staged tiles per warp (set at launch from the tile size)
  // A programmatic dependent of the append kernel just before it on the
  // stream (the one-call decode step): the CTAs may start while the append
  // runs.  kPdlAll: every CTA loads q and builds its tables, then waits for
  // the append's completion (griddepcontrol.wait) before reading the cache.
  // kPdlTail: this step's append writes nothing below t_tail (ring slots, a
  // value row or key group inside the tail), so the packed splits never wait
  // and only the tail's readers do.  kPdlOverlap: see below.  0: an
  // ordinary launch.
  int pdl;
};

// kPdlOverlap: launched after other work on the stream that writes neither
// q nor the cache (for instance another attention call): the CTAs read the
// cache and q at once; before a group's first workspace write they wait
// (bounded) until the previous call on this workspace has published the
// group's epoch, so that only the calls on the same workspace are ordered.
enum : int { kPdlAll = 1, kPdlTail = 2, kPdlOverlap = 3 };

// Programmatic dependent launch (sm_90+).  The primary kernel lets its
// dependent start early; the dependent waits for the primary's completion and
// memory visibility before touching what the primary writes.  Both are no-ops
// when the launch has no programmatic dependency.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a, const SeqLens& lens,
                             cudaStream_t st);
// One CTA runs the attention's bounded mbarrier wait on a phase that nothing
// completes and ORs 1 into *status (device memory) when it gives up.
cudaError_t launch_wait_probe(int* status, cudaStream_t st);

}  // namespace kivi
