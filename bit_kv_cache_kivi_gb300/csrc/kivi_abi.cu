// kivi_abi.cu -- host side of the C ABI declared in include/kivi.h:
// configuration checks, the residual policy (a pure function of the length,
// so no device readback is ever needed), the context-split policy, and the
// kernel launches.
#include <math.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/kivi.h"
#include "kivi_internal.cuh"

#define KIVI_API extern "C" __attribute__((visibility("default")))

struct kivi_cache {
  kivi_config cfg;
  kivi_buffers buf;
  int length;               // every sequence's length while `uniform`
  int uniform;              // 1: all sequences share `length`; 0: see lens
  int* lens;                // [batch] per-sequence lengths while !uniform
  int splits_override;      // 0 = automatic
  int overlap;              // kivi_set_attention_overlap
  const void* ws_ready;     // workspace whose counter area is known to be zero
  int device;               // the buffers' device (kNoDevice until the first launching call)
};

namespace {

thread_local int g_last_cuda_error = 0;

kivi_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KIVI_OK;
  g_last_cuda_error = (int)e;
  return KIVI_ECUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int kNoDevice = -1;   // not yet known
constexpr int kAnyDevice = -2;  // managed buffers: reachable from every device

// A caller buffer that the kernels, launched on `device`, may read or write
// directly: device memory of that device, managed memory, or page-locked
// host memory, which unified addressing maps into the device's address space
// at the same address (on a GB300 node the kernels then reach it over
// NVLink-C2C, with no staging copy).  Pageable host memory and another
// device's memory are refused before any launch.  Host only; no device work.
bool device_accessible(const void* p, int device) {
  cudaPointerAttributes at;
  const cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // do not leave the error for the next launch check
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == device;
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return at.devicePointer == p;
    default: return false;
  }
}

kivi_status check_config(const kivi_config* c) {
  if (!c) return KIVI_EINVAL;
  if (c->bits != 2 && c->bits != 3 && c->bits != 4 && c->bits != 8) return KIVI_EINVAL;
  if (c->group != kivi::kGroup || c->head_dim != kivi::kHeadDim) return KIVI_EINVAL;
  if (c->residual <= 0 || c->residual % c->group) return KIVI_ESHAPE;
  if (c->batch <= 0 || c->n_kv_heads <= 0 || c->n_q_heads <= 0) return KIVI_ESHAPE;
  if (c->n_q_heads % c->n_kv_heads) return KIVI_ESHAPE;
  if (c->max_tokens <= 0 || c->max_tokens % c->residual) return KIVI_ESHAPE;
  if (c->batch > 65535 || c->n_kv_heads > 4096) return KIVI_ESHAPE;  // grid limits
  // the attention grid's y extent: kv-heads x chunks of kHeadChunk query heads
  if ((long)c->n_kv_heads * ((c->n_q_heads / c->n_kv_heads + kivi::kHeadChunk - 1) / kivi::kHeadChunk) > 65535)
    return KIVI_ESHAPE;
  if (c->policy != KIVI_POLICY_ALG1 && c->policy != KIVI_POLICY_SHARED) return KIVI_EINVAL;
  if (c->outlier_channels < 0 || c->outlier_channels > kivi::kMaxOutliers) return KIVI_EINVAL;
  return KIVI_OK;
}

// The calling thread's current device, which must be the one holding the
// cache's buffers (found from the tile buffer on the first launching call):
// KIVI_EINVAL otherwise, before any launch.
kivi_status launch_device(kivi_cache* c, int* device) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return KIVI_ECUDA;
  }
  if (c->device == kNoDevice) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, c->buf.tiles) != cudaSuccess) {
      cudaGetLastError();
      return KIVI_EINVAL;
    }
    if (at.type == cudaMemoryTypeDevice) c->device = at.device;
    else if (at.type == cudaMemoryTypeManaged) c->device = kAnyDevice;
    else return KIVI_EINVAL;  // the cache itself must live in device memory
  }
  if (c->device != kAnyDevice && c->device != d) return KIVI_EINVAL;
  *device = d;
  return KIVI_OK;
}

// Sequence b's length.
int len_of(const kivi_cache* c, int b) { return c->uniform ? c->length : c->lens[b]; }

// The longest sequence.
int max_len(const kivi_cache* c) {
  if (c->uniform) return c->length;
  int m = 0;
  for (int b = 0; b < c->cfg.batch; ++b) m = c->lens[b] > m ? c->lens[b] : m;
  return m;
}

// The lengths as a launch parameter, for a launch that appends n tokens to
// every sequence.
void seq_lens(const kivi_cache* c, kivi::SeqLens* out, int n = 0) {
  out->uniform = c->uniform ? c->length : -1;
  out->n = n;
  if (c->uniform) {
    const int l = c->length, R = c->cfg.residual, p = c->cfg.policy;
    out->u_nq[0] = kivi::policy_nq_k(l, R, p);
    out->u_nq[1] = kivi::policy_nq_v(l, R, p);
    out->u_nq[2] = kivi::policy_nq_k(l + n, R, p);
    out->u_nq[3] = kivi::policy_nq_v(l + n, R, p);
  } else {
    for (int b = 0; b < c->cfg.batch; ++b) out->l[b] = c->lens[b];
  }
}

// Every sequence grows by n (host state after a successful launch).
void grow(kivi_cache* c, int n) {
  if (c->uniform) {
    c->length += n;
  } else {
    for (int b = 0; b < c->cfg.batch; ++b) c->lens[b] += n;
  }
}

// Set the lengths from a host array (uniform when they are all equal).
void set_lens(kivi_cache* c, const int* l) {
  bool same = true;
  for (int b = 1; b < c->cfg.batch; ++b) same = same && l[b] == l[0];
  c->uniform = same ? 1 : 0;
  c->length = same ? l[0] : -1;
  if (!same)
    for (int b = 0; b < c->cfg.batch; ++b) c->lens[b] = l[b];
}

// Ring slots: R under ALG1, R + G under SHARED (up to R + G - 1 fp16 tokens).
int ring_slots(const kivi_config& c) {
  return c.policy == KIVI_POLICY_SHARED ? c.residual + c.group : c.residual;
}

kivi::CacheView view(const kivi_cache* c) {
  kivi::CacheView v;
  v.tiles = static_cast<uint8_t*>(c->buf.tiles);
  v.ring_k = static_cast<__half*>(c->buf.ring_k);
  v.ring_v = static_cast<__half*>(c->buf.ring_v);
  v.B = c->cfg.batch;
  v.H = c->cfg.n_kv_heads;
  v.R = c->cfg.residual;
  v.W = ring_slots(c->cfg);
  v.Tcap = c->cfg.max_tokens;
  v.bits = c->cfg.bits;
  v.policy = c->cfg.policy;
  v.n_out = c->cfg.outlier_channels;
  v.tile_bytes = 2 * c->cfg.group * (c->cfg.head_dim * c->cfg.bits / 8) + 8 * c->cfg.head_dim +
                 kivi::outlier_block_bytes(c->cfg.outlier_channels);
  return v;
}

// Work units of the attention grid besides the split: (b, kv-head, chunk of
// kHeadChunk query heads).
long attention_units(const kivi_config& c) {
  const int grp = c.n_q_heads / c.n_kv_heads;
  return (long)c.batch * c.n_kv_heads * ((grp + kivi::kHeadChunk - 1) / kivi::kHeadChunk);
}

// Tail splits at most: the tail [floor32(nq_v), l) holds fewer than R + 32
// tokens under either policy.
int max_tail_splits(const kivi_config& c) {
  return (c.residual + 31 + kivi::kTailTok - 1) / kivi::kTailTok;
}

// Splits per attention unit in one wave of kivi::attn_ctas_per_sm CTAs per
// SM of a GB300, capped so that the partials merge in at most two levels.
int split_budget(const kivi_config& c) {
  const long u = attention_units(c);
  const int nb = kivi::attn_key_blocks(c.n_q_heads / c.n_kv_heads);
  long s = (long)kivi::attn_ctas_per_sm(c.bits, nb) * kivi::kTargetSMs / u;
  if (s > kivi::kMaxSplits) s = kivi::kMaxSplits;
  return (int)s;
}

// Upper bound on the packed-tile splits at any length: what the budget leaves
// beside the tail splits of a length with the fewest (one), at least one,
// and at most one per 32-token tile.
int max_tile_splits(const kivi_config& c) {
  long s = split_budget(c) - 1;
  if (s < 1) s = 1;
  const long by_len = (c.max_tokens + 31) / 32;
  return (int)(s < by_len ? s : by_len);
}

int max_splits(const kivi_config& c) {
  const int a = max_tail_splits(c) + 1, b = 1 + max_tile_splits(c);
  return a > b ? a : b;
}

// The cache's split configuration (kivi::make_plan plans one length with it).
// Launches that overlap the attention launch before them (`overlapped`)
// take a third of the budget and at least 128 tiles per packed split, and a
// tail of one split rides on the last packed split: the CTAs of several
// consecutive launches share the SMs, and the cost that every split pays
// once (its q tables, the wait for its first tile, its share of the merge)
// weighs more than the CTAs a launch leaves idle.  Measured on a GB300 with
// overlapped launches (per-group generations, no launch-wide waits): the
// Llama-3-8B decode shape (8 units of 127 tiles per sequence) takes 7.1 us
// with one packed split per unit carrying the tail, 7.8 us with two, 9.1 us
// with four; 131k tokens (4092 tiles, 8 units) 21.5 us with 23 packed
// splits, 22.2 us with 36, 22.5 us with 10 (its three tail splits stay
// separate).
// Tiles fewer for the packed split that carries a fused tail in overlapped
// plans: its fp16 tail round runs after its tiles.  Measured on the
// Llama-3-8B decode shape (2 packed splits of 127 tiles per unit): 8.6 us
// per launch with even splits, 8.1 us with 72 + 55 tiles (a discount of 32
// or 40), 8.6 us again with 96 + 31.
constexpr int kFusedDiscount = 32;

kivi::SplitCfg split_cfg(const kivi_cache* c, bool overlapped) {
  kivi::SplitCfg sc;
  const int budget = split_budget(c->cfg);
  sc.budget = overlapped ? (budget / 3 > 1 ? budget / 3 : 1) : budget;
  sc.min_tiles = overlapped ? 128 : 8;
  sc.fuse_single_tail = overlapped ? 1 : 0;
  sc.fused_discount = overlapped ? kFusedDiscount : 0;
  sc.max_splits = max_splits(c->cfg);
  sc.override_splits = c->splits_override;
  return sc;
}

kivi::SeqPlan plan_of(const kivi_cache* c, int l, bool overlapped) {
  return kivi::make_plan(l, c->cfg.residual, c->cfg.policy, split_cfg(c, overlapped));
}

// Workspace layout (attention group gid = (b, kv-head, head chunk), S = max
// splits, G = ceil(S / kMergeGroup), C = kHeadChunk):
//   partial outputs [gid][S][C][D] f32, partial (max, sum) [gid][S][C][2] f32,
//   group outputs [gid][G][C][D] f32, group (max, sum) [gid][G][C][2] f32,
//   split-group counters [gid][G] int, group counters [gid] int, then a
//   16-byte slot whose first int is the status word (nonzero after a
//   timed-out wait).
struct WsLayout {
  size_t o_off, ml_off, o1_off, ml1_off, cnt_off, cnt2_off, epoch_off, status_off, total;
  int groups;
};

WsLayout ws_layout(const kivi_config& c) {
  const size_t units = (size_t)attention_units(c);
  const size_t S = (size_t)max_splits(c);
  const size_t G = (S + kivi::kMergeGroup - 1) / kivi::kMergeGroup;
  const size_t C = kivi::kHeadChunk, D = (size_t)c.head_dim;
  WsLayout w;
  w.groups = (int)G;
  w.o_off = 0;
  w.ml_off = w.o_off + units * S * C * D * 4;
  w.o1_off = w.ml_off + units * S * C * 2 * 4;
  w.ml1_off = w.o1_off + units * G * C * D * 4;
  w.cnt_off = w.ml1_off + units * G * C * 2 * 4;
  w.cnt2_off = w.cnt_off + units * G * 4;
  w.epoch_off = w.cnt2_off + units * 4;
  w.status_off = (w.epoch_off + units * 8 + 15) / 16 * 16;
  w.total = w.status_off + 16;
  return w;
}

}  // namespace

KIVI_API kivi_status kivi_cache_sizes(const kivi_config* cfg, size_t bytes[3]) {
  kivi_status st = check_config(cfg);
  if (st != KIVI_OK) return st;
  if (!bytes) return KIVI_EINVAL;
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  const size_t T = cfg->max_tokens, D = cfg->head_dim, G = cfg->group;
  // a tile: key and value code rows of G tokens, key scale / zero [D], value
  // scale / zero [G][D / G] (f16)
  const size_t tile = 2 * G * (D * cfg->bits / 8) + 4 * D * 2 +
                      (size_t)kivi::outlier_block_bytes(cfg->outlier_channels);
  bytes[0] = units * (T / G) * tile;            // tiles
  bytes[1] = units * ring_slots(*cfg) * D * 2;  // ring_k
  bytes[2] = bytes[1];                          // ring_v
  return KIVI_OK;
}

KIVI_API kivi_status kivi_cache_init(const kivi_config* cfg, const kivi_buffers* bufs,
                                     kivi_cache** out) {
  if (!out) return KIVI_EINVAL;
  *out = nullptr;
  kivi_status st = check_config(cfg);
  if (st != KIVI_OK) return st;
  if (!bufs) return KIVI_EINVAL;
  const void* ptrs[3] = {bufs->tiles, bufs->ring_k, bufs->ring_v};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KIVI_EINVAL;
  kivi_cache* c = static_cast<kivi_cache*>(calloc(1, sizeof(kivi_cache)));
  if (!c) return KIVI_EINVAL;
  c->lens = static_cast<int*>(calloc((size_t)cfg->batch, sizeof(int)));
  if (!c->lens) {
    free(c);
    return KIVI_EINVAL;
  }
  c->cfg = *cfg;
  c->buf = *bufs;
  c->uniform = 1;
  c->device = kNoDevice;
  *out = c;
  return KIVI_OK;
}

namespace {

bool dtype_ok(kivi_dtype d) { return d == KIVI_F32 || d == KIVI_F16 || d == KIVI_BF16; }

// Prefill of an empty cache; lens = nullptr: every sequence takes t_in tokens.
kivi_status prefill(kivi_cache* c, const void* k, const void* v, kivi_dtype dtype, int t_in, const int* lens,
                    void* stream) {
  if (!c) return KIVI_EINVAL;
  if (!dtype_ok(dtype)) return KIVI_EDTYPE;
  if (c->uniform ? c->length != 0 : true) return KIVI_ESTATE;
  if (t_in < 0) return KIVI_ESHAPE;
  const int B = c->cfg.batch;
  if (lens) {
    for (int b = 0; b < B; ++b) {
      if (lens[b] < 0 || lens[b] > c->cfg.max_tokens) return KIVI_ECAPACITY;
      if (lens[b] > t_in) return KIVI_ESHAPE;
    }
    bool same = true;
    for (int b = 1; b < B; ++b) same = same && lens[b] == lens[0];
    if (!same && B > kivi::kMaxVarBatch) return KIVI_ESHAPE;
  } else if (t_in > c->cfg.max_tokens) {
    return KIVI_ECAPACITY;
  }
  if (t_in == 0) return KIVI_OK;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return KIVI_EINVAL;
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(k, dev) || !device_accessible(v, dev)) return KIVI_EINVAL;
  kivi_cache tmp = *c;  // the lengths the launch will produce
  if (lens) set_lens(&tmp, lens);
  else tmp.length = t_in;
  kivi::SeqLens sl;
  seq_lens(&tmp, &sl);
  kivi_status st = cuda_status(kivi::launch_quantize_prefill(view(c), k, v, (int)dtype, t_in, sl,
                                                             static_cast<cudaStream_t>(stream)));
  if (st != KIVI_OK) return st;
  if (lens) set_lens(c, lens);
  else c->length = t_in;
  return KIVI_OK;
}

}  // namespace

KIVI_API kivi_status kivi_quantize_prefill(kivi_cache* c, const void* k, const void* v,
                                           kivi_dtype dtype, int n_tokens, void* stream) {
  return prefill(c, k, v, dtype, n_tokens, nullptr, stream);
}

KIVI_API kivi_status kivi_quantize_prefill_varlen(kivi_cache* c, const void* k, const void* v,
                                                  kivi_dtype dtype, int max_len, const int* lengths,
                                                  void* stream) {
  if (!c || !lengths) return KIVI_EINVAL;
  return prefill(c, k, v, dtype, max_len, lengths, stream);
}

namespace {

// The argument checks of a one-token append (before any launch).
kivi_status append_checks(const kivi_cache* c, const void* k_new, const void* v_new, kivi_dtype dtype) {
  if (!c) return KIVI_EINVAL;
  if (!dtype_ok(dtype)) return KIVI_EDTYPE;
  if (!k_new || !v_new) return KIVI_EINVAL;
  if (max_len(c) >= c->cfg.max_tokens) return KIVI_ECAPACITY;
  if (c->cfg.policy == KIVI_POLICY_SHARED && (!aligned16(k_new) || !aligned16(v_new))) return KIVI_EINVAL;
  return KIVI_OK;
}

// The launches of a checked one-token append; the lengths grow on success.
// trig: the append lets the launch after it (a decode step's attention)
// start at once; 0: nothing starts before the append completes (see
// kivi::launch_append).
kivi_status append_launch(kivi_cache* c, const void* k_new, const void* v_new, kivi_dtype dtype, void* stream,
                          int trig = 0) {
  kivi::SeqLens sl;
  seq_lens(c, &sl, 1);
  cudaError_t e;
  if (c->cfg.policy == KIVI_POLICY_SHARED) {
    // the one-token case of the multi-token append: a whole group of keys and
    // values is quantized when nq grows, then the token goes to the ring
    e = kivi::launch_append_tokens(view(c), k_new, v_new, (int)dtype, 1, sl, static_cast<cudaStream_t>(stream),
                                   trig);
  } else {
    e = kivi::launch_append(view(c), k_new, v_new, (int)dtype, sl, static_cast<cudaStream_t>(stream), trig);
  }
  kivi_status st = cuda_status(e);
  if (st == KIVI_OK) grow(c, 1);
  return st;
}

}  // namespace

KIVI_API kivi_status kivi_append_decode(kivi_cache* c, const void* k_new, const void* v_new,
                                        kivi_dtype dtype, void* stream) {
  const kivi_status chk = append_checks(c, k_new, v_new, dtype);
  if (chk != KIVI_OK) return chk;
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(k_new, dev) || !device_accessible(v_new, dev)) return KIVI_EINVAL;
  return append_launch(c, k_new, v_new, dtype, stream);
}

KIVI_API kivi_status kivi_append_tokens(kivi_cache* c, const void* k, const void* v, kivi_dtype dtype,
                                        int n_tokens, void* stream) {
  if (!c) return KIVI_EINVAL;
  if (!dtype_ok(dtype)) return KIVI_EDTYPE;
  if (n_tokens <= 0 || !k || !v || !aligned16(k) || !aligned16(v)) return KIVI_EINVAL;
  if ((long)max_len(c) + n_tokens > c->cfg.max_tokens) return KIVI_ECAPACITY;
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(k, dev) || !device_accessible(v, dev)) return KIVI_EINVAL;
  kivi::SeqLens sl;
  seq_lens(c, &sl, n_tokens);
  kivi_status st = cuda_status(
      kivi::launch_append_tokens(view(c), k, v, (int)dtype, n_tokens, sl, static_cast<cudaStream_t>(stream)));
  if (st == KIVI_OK) grow(c, n_tokens);
  return st;
}

KIVI_API kivi_status kivi_cache_set_length(kivi_cache* c, int length) {
  if (!c) return KIVI_EINVAL;
  if (length < 0 || length > c->cfg.max_tokens) return KIVI_ECAPACITY;
  c->uniform = 1;
  c->length = length;
  return KIVI_OK;
}

KIVI_API kivi_status kivi_cache_set_lengths(kivi_cache* c, const int* lengths) {
  if (!c || !lengths) return KIVI_EINVAL;
  bool same = true;
  for (int b = 0; b < c->cfg.batch; ++b) {
    if (lengths[b] < 0 || lengths[b] > c->cfg.max_tokens) return KIVI_ECAPACITY;
    same = same && lengths[b] == lengths[0];
  }
  if (!same && c->cfg.batch > kivi::kMaxVarBatch) return KIVI_ESHAPE;
  set_lens(c, lengths);
  return KIVI_OK;
}

KIVI_API kivi_status kivi_cache_lengths(const kivi_cache* c, int* lengths) {
  if (!c || !lengths) return KIVI_EINVAL;
  for (int b = 0; b < c->cfg.batch; ++b) lengths[b] = len_of(c, b);
  return KIVI_OK;
}

KIVI_API size_t kivi_attention_workspace_bytes(const kivi_cache* c) {
  if (!c) return 0;
  return ws_layout(c->cfg).total;
}

KIVI_API kivi_status kivi_set_attention_splits(kivi_cache* c, int n_splits) {
  if (!c || n_splits < 0) return KIVI_EINVAL;
  c->splits_override = n_splits;
  return KIVI_OK;
}

KIVI_API int kivi_attention_splits(const kivi_cache* c, int l) {
  if (!c || l <= 0) return 0;
  return plan_of(c, l, c->overlap != 0).splits;
}

namespace {

// The attention launch arguments that depend on the lengths and the
// workspace; KIVI_ESTATE when some sequence is empty.
kivi_status attn_args(const kivi_cache* c, const void* q, kivi_dtype q_dtype, void* out, float softmax_scale,
                      char* ws, bool overlapped, kivi::AttnArgs* a, kivi::SeqLens* sl) {
  const int B = c->cfg.batch;
  for (int b = 0; b < (c->uniform ? 1 : B); ++b)
    if (len_of(c, b) <= 0) return KIVI_ESTATE;
  a->q = q;
  a->out = out;
  a->q_dtype = (int)q_dtype;
  a->Hq = c->cfg.n_q_heads;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)c->cfg.head_dim);
  a->scale_log2 = scale * 1.4426950408889634f;
  a->scfg = split_cfg(c, overlapped);
  seq_lens(c, sl);
  if (c->uniform) {
    a->plan = plan_of(c, c->length, overlapped);
    a->splits = a->plan.splits;
  } else {
    a->plan = plan_of(c, c->lens[0], overlapped);
    a->splits = 0;
    for (int b = 0; b < B; ++b) {
      const int s = plan_of(c, c->lens[b], overlapped).splits;
      a->splits = s > a->splits ? s : a->splits;
    }
  }
  const WsLayout w = ws_layout(c->cfg);
  a->ws_o = reinterpret_cast<float*>(ws + w.o_off);
  a->ws_ml = reinterpret_cast<float*>(ws + w.ml_off);
  a->ws_o1 = reinterpret_cast<float*>(ws + w.o1_off);
  a->ws_ml1 = reinterpret_cast<float*>(ws + w.ml1_off);
  a->merge_groups = w.groups;
  a->counters = reinterpret_cast<int*>(ws + w.cnt_off);
  a->counters2 = reinterpret_cast<int*>(ws + w.cnt2_off);
  a->status = reinterpret_cast<int*>(ws + w.status_off);
  a->epochs = reinterpret_cast<unsigned*>(ws + w.epoch_off);
  a->epoch_on = 0;
  a->pdl = 0;
  return KIVI_OK;
}

}  // namespace

KIVI_API kivi_status kivi_decode_attention(kivi_cache* c, const void* q, kivi_dtype q_dtype,
                                           void* out, float softmax_scale, void* workspace,
                                           size_t ws_bytes, void* stream) {
  if (!c) return KIVI_EINVAL;
  if (!dtype_ok(q_dtype)) return KIVI_EDTYPE;
  if (!q || !out) return KIVI_EINVAL;
  if (c->uniform && c->length <= 0) return KIVI_ESTATE;
  if (!workspace || !aligned16(workspace) || ws_bytes < kivi_attention_workspace_bytes(c))
    return KIVI_EWORKSPACE;
  kivi::AttnArgs a;
  kivi::SeqLens sl;
  kivi_status ast = attn_args(c, q, q_dtype, out, softmax_scale, static_cast<char*>(workspace), c->overlap != 0, &a, &sl);
  if (ast != KIVI_OK) return ast;
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(q, dev) || !device_accessible(out, dev)) return KIVI_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->ws_ready != workspace) {
    if (!device_accessible(workspace, dev)) return KIVI_EWORKSPACE;
    const WsLayout w = ws_layout(c->cfg);
    kivi_status z = cuda_status(cudaMemsetAsync(a.counters, 0, w.total - w.cnt_off, st));
    if (z != KIVI_OK) return z;
    c->ws_ready = workspace;
  }
  if (c->overlap) a.pdl = kivi::kPdlOverlap;
  a.epoch_on = 1;  // every call on the cache's workspace keeps its generations
  return cuda_status(kivi::launch_attention(view(c), a, sl, st));
}

KIVI_API kivi_status kivi_set_attention_overlap(kivi_cache* c, int enable) {
  if (!c || (enable != 0 && enable != 1)) return KIVI_EINVAL;
  c->overlap = enable;
  return KIVI_OK;
}

KIVI_API kivi_status kivi_decode_step(kivi_cache* c, const void* k_new, const void* v_new,
                                      kivi_dtype kv_dtype, const void* q, kivi_dtype q_dtype, void* out,
                                      float softmax_scale, void* workspace, size_t ws_bytes,
                                      void* stream) {
  // every check of both halves before any launch
  const kivi_status chk = append_checks(c, k_new, v_new, kv_dtype);
  if (chk != KIVI_OK) return chk;
  if (!dtype_ok(q_dtype)) return KIVI_EDTYPE;
  if (!q || !out) return KIVI_EINVAL;
  if (!workspace || !aligned16(workspace) || ws_bytes < kivi_attention_workspace_bytes(c))
    return KIVI_EWORKSPACE;
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(k_new, dev) || !device_accessible(v_new, dev) || !device_accessible(q, dev) ||
      !device_accessible(out, dev))
    return KIVI_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->ws_ready != workspace) {
    if (!device_accessible(workspace, dev)) return KIVI_EWORKSPACE;
    // before the append, so that the attention's only predecessor is the append
    const WsLayout w = ws_layout(c->cfg);
    kivi_status z =
        cuda_status(cudaMemsetAsync(static_cast<char*>(workspace) + w.cnt_off, 0, w.total - w.cnt_off, st));
    if (z != KIVI_OK) return z;
    c->ws_ready = workspace;
  }
  // the append lets the attention start at once (its prologue, and the
  // packed splits on most steps, run beside the append)
  kivi_status s1 = append_launch(c, k_new, v_new, kv_dtype, stream, 1);
  if (s1 != KIVI_OK) return s1;
  kivi::AttnArgs a;
  kivi::SeqLens sl;
  kivi_status ast = attn_args(c, q, q_dtype, out, softmax_scale, static_cast<char*>(workspace), false, &a, &sl);
  if (ast != KIVI_OK) return ast;  // not reached: every sequence holds a token now
  // Which tiles did the append write?  Under either policy, the only write
  // below t_tail = 32 floor(nq_v(l) / 32) is on a step where l - R reaches a
  // multiple of G: the value row leaving the window (Algorithm 1) or the
  // group just quantized (shared window) then closes the last packed tile.
  // On every other step the append writes ring slots and rows or key groups
  // of the tail alone, and the packed splits need not wait for it.
  bool packed_untouched = true;
  for (int b = 0; b < (c->uniform ? 1 : c->cfg.batch); ++b) {
    const int l = len_of(c, b);
    if (l > c->cfg.residual && (l - c->cfg.residual) % c->cfg.group == 0) packed_untouched = false;
  }
  a.pdl = packed_untouched ? kivi::kPdlTail : kivi::kPdlAll;
  a.epoch_on = 1;
  return cuda_status(kivi::launch_attention(view(c), a, sl, st));
}

KIVI_API int kivi_cache_length(const kivi_cache* c) {
  if (!c) return -1;
  return c->uniform ? c->length : -2;
}

KIVI_API kivi_status kivi_cache_reset(kivi_cache* c) {
  if (!c) return KIVI_EINVAL;
  c->uniform = 1;
  c->length = 0;
  return KIVI_OK;
}

KIVI_API void kivi_cache_destroy(kivi_cache* c) {
  if (!c) return;
  free(c->lens);
  free(c);
}

KIVI_API const char* kivi_status_string(kivi_status s) {
  switch (s) {
    case KIVI_OK: return "ok";
    case KIVI_EINVAL: return "invalid argument (null, unsupported parameter or misaligned buffer)";
    case KIVI_ESHAPE: return "inconsistent shape";
    case KIVI_ECAPACITY: return "cache capacity exceeded";
    case KIVI_EDTYPE: return "unknown dtype";
    case KIVI_ECUDA: return "CUDA launch error";
    case KIVI_ESTATE: return "invalid in the cache's current state";
    case KIVI_EWORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

KIVI_API int kivi_last_cuda_error(void) { return g_last_cuda_error; }

// The attention's bounded wait on a barrier phase nothing completes: the
// probe returns after the wait limit with 1 ORed into *status.
KIVI_API kivi_status kivi_check_bounded_wait(int* status, void* stream) {
  if (!status || ((uintptr_t)status & 3u)) return KIVI_EINVAL;
  int dev = 0;
  const kivi_status ds = cuda_status(cudaGetDevice(&dev));
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(status, dev)) return KIVI_EINVAL;
  return cuda_status(kivi::launch_wait_probe(status, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// Decode attention without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: a plugin inside a host framework whose device memory is handed
// out only by that framework's own pool, or a latency-critical path that must
// not pay cudaMalloc's implicit device-wide synchronization.  For them the
// library keeps one fixed scratch area in device global memory, declared
// below, and kivi_decode_attention_static uses it instead of a workspace
// argument.  Every GPU that loads this library holds the area until the
// process exits.

static __device__ __align__(256) unsigned char g_static_ws[KIVI_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices];  // device address of g_static_ws, per device

// Device address of the scratch area on the current device, looked up once
// per device (the symbol's host-side name is not a device address).
cudaError_t static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace

KIVI_API kivi_status kivi_decode_attention_static(kivi_cache* c, const void* q,
                                                  kivi_dtype q_dtype, void* out,
                                                  float softmax_scale, void* stream) {
  if (!c) return KIVI_EINVAL;
  if (q_dtype != KIVI_F32 && q_dtype != KIVI_F16 && q_dtype != KIVI_BF16) return KIVI_EDTYPE;
  if (!q || !out) return KIVI_EINVAL;
  if (c->uniform && c->length <= 0) return KIVI_ESTATE;
  const WsLayout w = ws_layout(c->cfg);
  if (w.total > (size_t)KIVI_STATIC_WORKSPACE_BYTES) return KIVI_EWORKSPACE;
  // every check first, so that a refused call does no CUDA work (the area's
  // address lookup may load the module on the current device)
  int dev = 0;
  const kivi_status ds = launch_device(c, &dev);
  if (ds != KIVI_OK) return ds;
  if (!device_accessible(q, dev) || !device_accessible(out, dev)) return KIVI_EINVAL;
  for (int b = 0; b < (c->uniform ? 1 : c->cfg.batch); ++b)
    if (len_of(c, b) <= 0) return KIVI_ESTATE;
  void* ws = nullptr;
  kivi_status st = cuda_status(static_ws_address(&ws));
  if (st != KIVI_OK) return st;
  kivi::AttnArgs a;
  kivi::SeqLens sl;
  st = attn_args(c, q, q_dtype, out, softmax_scale, static_cast<char*>(ws), false, &a, &sl);
  if (st != KIVI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The area keeps whatever the previous call left; the split counters must
  // start at zero, so clear them on every call (a memset, not an allocation).
  st = cuda_status(cudaMemsetAsync(a.counters, 0, w.total - w.cnt_off, s));
  if (st != KIVI_OK) return st;
  return cuda_status(kivi::launch_attention(view(c), a, sl, s));
}
