/*
 * kivi.h -- C ABI of the GB300 (sm_103a) KIVI KV-cache library.
 *
 * KIVI keeps the KV cache of a decoder in low-bit codes (2, 3, 4 or 8 bits): keys are
 * quantized per channel (groups of G tokens along the token axis), values
 * per token (groups of G channels), each group with an fp16 scale and zero
 * point; the most recent tokens stay in an fp16 residual window.  Decode
 * attention reads the packed cache directly.
 *
 * Sources (page title, section):
 *   - veloxquant-mlx docs, "KIVI", "How it works" items 1-4 and the
 *     zero/scale/q/recon formulas (quantizer, grouping axes, residual
 *     window, group-aligned flushes);
 *   - chooblog review "KIVI: A Tuning-Free Asymmetric 2bit Quantization for
 *     KV Cache (ICML'24)", §1.1 (quantization definition), §1.3 (prefill and
 *     decoding phases: cache X_K, X_V; append t_K, t_V; softmax(t_Q X_K^T) X_V),
 *     §3.2.2-3.2.3 (grouped + residual split, Algorithm 1), §3.2
 *     "System-Level" (dequantization fused with the matrix product);
 *   - "KIVI - 2-bit KV cache quantisation" notebook (attention scaled by
 *     1/sqrt(head_dim); fp16 (min, scale) pair per group).
 *
 * Conventions shared by every call
 *   - Device memory is owned by the caller; the library never allocates
 *     device memory.  It allocates only the small host handle.
 *   - Inputs and outputs passed per call (k, v, k_new, v_new, q, out) may be
 *     device memory or page-locked host memory (cudaHostAlloc /
 *     cudaHostRegister): under unified addressing the kernels read and write
 *     such host buffers directly (on a GB300 node over NVLink-C2C), with no
 *     staging copy.  Pageable host memory is refused with KIVI_EINVAL before
 *     any launch (checked with cudaPointerGetAttributes).
 *   - Calls that launch work must be made with the device that holds the
 *     cache's buffers current (the device is read from the tile buffer on
 *     the first such call), and device buffers passed per call (inputs,
 *     outputs, workspace) must live on that device; otherwise KIVI_EINVAL
 *     (KIVI_EWORKSPACE for the workspace) before any launch.
 *   - All work is asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  No call synchronizes the
 *     device or reads device memory back.
 *   - Shapes and state are checked on the host before any launch; a call
 *     that returns an error has launched nothing, except KIVI_ECUDA, which
 *     reports a launch error (see kivi_last_cuda_error).
 *   - A handle is not thread-safe; calls on one handle must be serialized
 *     by the caller (the stream orders the device work).
 *   - Supported by this library: bits 2, 3, 4 or 8, group 32, head_dim 128,
 *     residual a multiple of 32, any batch / head counts with
 *     n_q_heads a multiple of n_kv_heads.
 *   - Inputs must be finite and within the fp16 range; every input element
 *     is rounded to fp16 (nearest even) before it is quantized or stored.
 *
 * Storage layout (all buffers 16-byte aligned; B batch, H = n_kv_heads,
 * T = max_tokens, D = head_dim, G = group, R = residual, b = bits,
 * RB = D*b/8 bytes per packed row):
 *   tiles   [B][H][T/G] tiles of 2*G*RB + 8*D bytes: tile j holds all the
 *           quantized state of tokens [G*j, G*j + G) of a (batch, kv-head):
 *             [0, 2*D)             key zero [D] (f16; the tile's key group,
 *                                  one per channel)
 *             [2*D, 2*D + G*RB)    key code rows, token-major
 *             then                 value code rows, token-major (G*RB bytes)
 *             then f16 arrays:     key scale [D],
 *                                  value scale [G][D/G], value zero [G][D/G]
 *                                  (one per G channels per token)
 *           (the key zeros lead: the decode attention stages the rest of a
 *           tile with one bulk copy and reads the zeros of sixteen tiles at
 *           once for the term zero x q)
 *           With kivi_config.outlier_channels = n > 0, a tile ends with an
 *           outlier block of 16 + 64*n bytes: the n channel indices (u8,
 *           largest max |k| first, zero padded to 16 bytes), then
 *           value[G][n] (f16) -- the tile's fp16 outlier keys; those
 *           channels' codes, key scales and key zeros in the tile are 0.
 *           At 8 bits the code rows are stored rotated by whole 16-byte
 *           chunks (key row r by r & 1 chunks, value row r by 2*(r & 3);
 *           logical chunk c at chunk (c + rotation) mod 8), so that the
 *           attention kernel's shared-memory reads avoid bank conflicts.
 *           The f16 arrays are stored in the order the decode-attention
 *           tensor-core fragments take them (G = 32, D = 128):
 *             key scale / zero: 32-bit word i of pair block m holds channels
 *               (P*m + i, P*m + i + P/2), P = 16 at 2 and 3 bits, 8 at 4
 *               bits, 4 at 8 bits, i.e.
 *               channel c is at f16 slot P*(c/P) + 2*(c%(P/2)) + (c%P)/(P/2);
 *             value scale / zero: tokens (8a + r, 8a + r + 4), r < 4, share
 *               32-bit word 4*(4a + r) + g for group g, i.e. token t, group g
 *               is at f16 slot 32*(t/8) + 8*(t%4) + 2*g + (t/4)%2.
 *   ring_k  [B][H][W][D]     f16  residual keys, token t in slot t mod W
 *   ring_v  [B][H][W][D]     f16  residual values, token t in slot t mod W
 * Channel e of a key row is bits [(e*b)%8, (e*b)%8 + b) of byte (e*b)/8.
 * Value rows are group-interleaved in units of 4 channels (b/2 bytes): the
 * unit of channels G*g + 4*w .. +3 sits at unit position 4*w + g, its
 * channels in ascending bit order.  A tile is one contiguous block so that
 * decode attention stages it with a single bulk copy.
 * 3-bit rows (48 bytes; the pages print no 3-bit packing, so this is the
 * library's choice) are two planes: bytes [0, 32) hold the low two bits of
 * every code exactly as a 2-bit row, bytes [32, 48) the high bits in eight
 * 16-bit units.  Key unit 2*W + h (W < 4, h < 2) holds channels 16*m + 8*h
 * + i for m in {W, W + 4} and i < 8, with set s = m / 4; value unit w holds
 * channels 32*g + 4*w + c of the four groups g, with s = g / 2 and
 * i = 4*(g % 2) + c.  (s, i) sits at bit p = 2*(i%4) + 2 + (i >= 4) of its
 * unit, or (p + 8) % 16 when s = 1.
 * Residual policy (kivi_config.policy):
 *   KIVI_POLICY_ALG1 (the chooblog review's Algorithm 1): after l tokens the
 *     first nq_k(l) = R*floor(l/R) keys and the first nq_v(l) = max(l-R, 0)
 *     values are quantized; W = R ring slots.
 *   KIVI_POLICY_SHARED (veloxquant-mlx "KIVI" How it works, items 3-4: at
 *     least the R most recent tokens stay fp16, aged-out tokens are
 *     quantized in whole groups): keys and values share nq(l) =
 *     G*floor(max(l-R, 0)/G); W = R + G ring slots.
 * The rest of the tokens are in the rings.  Rows and slots that hold no live
 * token are left untouched.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KIVI_OK = 0,
  KIVI_EINVAL = 1,     /* null pointer, unsupported parameter, misaligned buffer */
  KIVI_ESHAPE = 2,     /* inconsistent sizes (divisibility, token counts) */
  KIVI_ECAPACITY = 3,  /* the cache would exceed max_tokens */
  KIVI_EDTYPE = 4,     /* unknown dtype code */
  KIVI_ECUDA = 5,      /* a kernel launch failed; see kivi_last_cuda_error() */
  KIVI_ESTATE = 6,     /* call not valid in the cache's current state */
  KIVI_EWORKSPACE = 7  /* workspace missing, misaligned or too small */
} kivi_status;

typedef enum { KIVI_F32 = 0, KIVI_F16 = 1, KIVI_BF16 = 2 } kivi_dtype;

typedef enum { KIVI_POLICY_ALG1 = 0, KIVI_POLICY_SHARED = 1 } kivi_policy;

/* Cache configuration (veloxquant-mlx "KIVI" usage: bit width, group size,
 * residual length) plus the tensor shape. */
typedef struct {
  int bits;        /* 2, 3, 4 or 8 */
  int group;       /* G: 32 in this library */
  int residual;    /* R: fp16 window, a multiple of G */
  int head_dim;    /* D: 128 in this library */
  int batch;       /* B */
  int n_kv_heads;  /* H */
  int n_q_heads;   /* a multiple of n_kv_heads; query head j reads KV head j/(Hq/H) */
  int max_tokens;  /* capacity T, a multiple of R */
  int policy;      /* kivi_policy: KIVI_POLICY_ALG1 (0) or KIVI_POLICY_SHARED */
  int outlier_channels; /* 0..4: per key group, this many channels with the
                         * largest max |k| stay fp16 (the "KIVI - 2-bit KV
                         * cache quantisation" notebook, Exercises item 2);
                         * 0 = plain KIVI */
} kivi_config;

/* The three caller-owned device buffers, in the layout above. */
typedef struct {
  void *tiles;
  void *ring_k, *ring_v;
} kivi_buffers;

typedef struct kivi_cache kivi_cache; /* opaque host handle */

/* Bytes each buffer needs, in kivi_buffers order.  Host only; no GPU.
 * Returns KIVI_EINVAL / KIVI_ESHAPE for a config this library rejects. */
kivi_status kivi_cache_sizes(const kivi_config *cfg, size_t bytes[3]);

/* Validate cfg, bind the buffers and create an empty handle (length 0).
 * Host only; the buffers' contents are not touched.  The buffers must stay
 * valid until kivi_cache_destroy. */
kivi_status kivi_cache_init(const kivi_config *cfg, const kivi_buffers *bufs,
                            kivi_cache **out);

/* Prefill (review §1.3 prefill phase; Algorithm 1 prefill steps B-D).
 * k, v: device [B][H][n_tokens][D] of dtype, contiguous.  The cache must be
 * empty (KIVI_ESTATE otherwise) and 0 <= n_tokens <= max_tokens.
 * Quantizes the first nq_k keys per channel and the first nq_v values per
 * token, stores the remaining tokens in the rings; length becomes n_tokens. */
kivi_status kivi_quantize_prefill(kivi_cache *c, const void *k, const void *v,
                                  kivi_dtype dtype, int n_tokens, void *stream);

/* Sequences of a batch may have different lengths (one per batch row; every
 * call below applies the policy to each sequence at its own length).  With
 * more than KIVI_MAX_VARLEN_BATCH sequences, all lengths must be equal. */
#define KIVI_MAX_VARLEN_BATCH 1024

/* Prefill with per-sequence lengths: k, v: device [B][H][max_len][D] of
 * dtype, contiguous, 16-byte aligned; sequence b is its first lengths[b]
 * rows (the others are ignored).  lengths: host int[B], each in [0,
 * max_tokens] (KIVI_ECAPACITY) and <= max_len (KIVI_ESHAPE).  The cache must
 * be empty.  Each sequence is quantized exactly as kivi_quantize_prefill
 * would quantize it alone. */
kivi_status kivi_quantize_prefill_varlen(kivi_cache *c, const void *k,
                                         const void *v, kivi_dtype dtype,
                                         int max_len, const int *lengths,
                                         void *stream);

/* Append one decoded token to every sequence (review §1.3 decoding step 1;
 * Algorithm 1 decoding phase).  k_new, v_new: device [B][H][D] of dtype.
 * Token t = the sequence's length goes to ring slot t mod W.  ALG1: if t >= R, the value token t-R leaves the
 * window and is quantized per token; if t+1 is a multiple of R, the R keys of
 * the ring (a whole number of groups) are quantized per channel.  SHARED:
 * when t+1-R reaches a positive multiple of G, the G oldest ring tokens are
 * quantized, keys per channel (one group) and values per token.  The
 * decision is taken on the host from the length alone.  KIVI_ECAPACITY when
 * the longest sequence is at max_tokens; under SHARED, KIVI_EINVAL unless
 * k_new and v_new are 16-byte aligned. */
kivi_status kivi_append_decode(kivi_cache *c, const void *k_new,
                               const void *v_new, kivi_dtype dtype,
                               void *stream);

/* Append n_tokens tokens at once to every sequence (chunked prefill into a
 * non-empty cache;
 * the review §1.3 prefill step continued on a cache that already holds
 * tokens).  k, v: device [B][H][n_tokens][D] of dtype, contiguous,
 * 16-byte aligned.  The result is the cache that n_tokens calls of
 * kivi_append_decode would leave (the review's Algorithm 1 applied token by
 * token), bit for bit: the key groups that become whole and the value tokens
 * that leave the window are quantized (old tokens read from the rings), then
 * the last min(n_tokens, R) tokens go to their ring slots.  Two kernel
 * launches on the stream.  KIVI_ECAPACITY if the longest sequence + n_tokens >
 * max_tokens, KIVI_EINVAL if n_tokens <= 0. */
kivi_status kivi_append_tokens(kivi_cache *c, const void *k, const void *v,
                               kivi_dtype dtype, int n_tokens, void *stream);

/* Declare the cache's length after its three buffers were restored from a
 * saved state (the buffers are the caller's tensors, so saving and restoring
 * a cache is copying them plus this length).
 * The length of a state is kivi_cache_length() at save time.  Host only; no
 * device work.  KIVI_ECAPACITY if length is outside [0, max_tokens]. */
kivi_status kivi_cache_set_length(kivi_cache *c, int length);

/* The same with per-sequence lengths (host int[B]); KIVI_ECAPACITY if one is
 * outside [0, max_tokens], KIVI_ESHAPE for unequal lengths past
 * KIVI_MAX_VARLEN_BATCH sequences.  Host only. */
kivi_status kivi_cache_set_lengths(kivi_cache *c, const int *lengths);

/* Per-sequence lengths into lengths (host int[B]).  Host only. */
kivi_status kivi_cache_lengths(const kivi_cache *c, int *lengths);

/* Device workspace (bytes) kivi_decode_attention needs for this handle's
 * shape at any length: split-K partial results, merged groups of partials,
 * counters, one epoch per (batch, kv-head, head chunk) for overlapping calls,
 * and a status word (the int at byte offset bytes - 16: bit 1 after a kernel
 * gave up waiting for its staged data, which only a device fault can cause;
 * bit 2 after an overlapping call gave up waiting for the previous call's
 * epoch, which only a broken contract can cause; it stays set until the
 * workspace is next cleared).  Host only. */
size_t kivi_attention_workspace_bytes(const kivi_cache *c);

/* Decode attention over the cache (review §1.3 decoding step 2:
 * out = softmax(q K^T * scale) V; §3.2 System-Level: dequantization fused
 * into the products).  q: device [B][n_q_heads][D] of q_dtype; out: device
 * [B][n_q_heads][D] of q_dtype.  softmax_scale <= 0 means 1/sqrt(D).
 * The context is split along the tokens; the CTA that finishes last in a
 * group of up to 16 splits of a (batch, kv-head) merges their partial (max,
 * sum, output) triples, and with more groups the last group merges the
 * groups, all in one kernel launch.
 * workspace: device, 16-byte aligned, ws_bytes >= kivi_attention_workspace_bytes.
 * It carries a small counter area between calls: the first call that sees a
 * given workspace pointer zeroes it (one cudaMemsetAsync on the stream) and
 * every call leaves it zero.  Do not write to the workspace between calls,
 * and do not share one workspace between calls that may overlap on the GPU.
 * Each sequence attends over its own length; KIVI_ESTATE when a sequence is
 * empty. */
kivi_status kivi_decode_attention(kivi_cache *c, const void *q,
                                  kivi_dtype q_dtype, void *out,
                                  float softmax_scale, void *workspace,
                                  size_t ws_bytes, void *stream);

/* One decode step (review §1.3 decoding phase: the new token's key and value
 * are concatenated to the cache, then out = softmax(q K^T * scale) V over all
 * l + 1 tokens): kivi_append_decode(c, k_new, v_new, kv_dtype) followed by
 * kivi_decode_attention(c, q, q_dtype, out, ...) on the same stream, with
 * the same arguments, layouts and results (bit for bit).
 * The attention is launched as a programmatic dependent of the append's last
 * kernel: its CTAs start while the append runs.  A CTA waits
 * (griddepcontrol.wait) for the append to complete before it reads anything
 * the append may have written: on a step where l - R reaches a multiple of
 * G (the append closes the last packed tile) every CTA builds its query
 * tables and then waits; on every other step only the CTAs that read the
 * fp16 tail wait, and the packed splits run beside the append.
 * The step's attention lets a launch after it start early only once its
 * append has completed, so that an overlapping attention call enqueued
 * after the step (kivi_set_attention_overlap) never reads a cache before the
 * step's write to it lands.  The step ignores the overlap setting.
 * Errors: every check of both halves is made before any launch (nothing runs
 * and the length is unchanged on KIVI_EINVAL, KIVI_EDTYPE, KIVI_ECAPACITY or
 * KIVI_EWORKSPACE).  If the append launches and the attention launch then
 * fails, the token stays appended (the length grows by one) and the call
 * returns KIVI_ECUDA. */
kivi_status kivi_decode_step(kivi_cache *c, const void *k_new,
                             const void *v_new, kivi_dtype kv_dtype,
                             const void *q, kivi_dtype q_dtype, void *out,
                             float softmax_scale, void *workspace,
                             size_t ws_bytes, void *stream);

/* Override the number of context splits (0 = automatic).  The first splits
 * always take the tail of the context that is still fp16 (plus the partial
 * value group before it), 64 tokens each; the others share the packed
 * 32-token tiles.  The automatic choice keeps the whole grid within one wave
 * of a 152-SM GB300 (four CTAs per SM; three at 4 bits with more than four
 * query heads per KV head, two at 8 bits), with at least eight tiles per
 * packed split and a multiple of four.  With the overlap on (see
 * kivi_set_attention_overlap) the automatic choice takes a third of that
 * budget and at least 128 tiles per packed split, and rides the tail on the last
 * packed split when the tail is a single split or the budget holds no tail
 * split beside it (that split then takes up to 32 tiles fewer): the CTAs of
 * consecutive launches then share the SMs, and fewer, longer splits pay the
 * fixed cost of a split (query tables, first tile, merge) fewer times.  An
 * override n asks for n splits in all, with or without the overlap; it is
 * clamped to the workspace bound, to one packed split per 32-token tile
 * and to at least one packed split. */
kivi_status kivi_set_attention_splits(kivi_cache *c, int n_splits);

/* Splits the next kivi_decode_attention call will use at length l (with the
 * handle's current overlap setting). */
int kivi_attention_splits(const kivi_cache *c, int l);

/* Let kivi_decode_attention calls on this handle overlap the kernel enqueued
 * just before them on the stream (enable = 1; 0, the default, turns it off;
 * KIVI_EINVAL for other values).  No counterpart on the pages: a launch-order
 * setting.  The attention is then launched as a programmatic dependent of
 * that kernel: its CTAs start as the earlier kernel's CTAs finish and read q
 * and the cache at once.  Calls on the same workspace are ordered by an
 * epoch per (batch, kv-head, head chunk) kept in the workspace: a call's CTAs
 * write the group's partials only once the previous call on that workspace
 * has finished with them (a bounded wait, see kivi_check_bounded_wait), and
 * the other CTAs do not wait for the kernel before.  A launch still
 * completes only after the one before it (one CTA waits for it last), so
 * whatever follows on the stream follows them all.
 * The contract:
 * - the work enqueued since the last launch that is not an overlapping
 *   attention call writes neither this call's q nor this cache
 *   (overlapping calls enqueued back to back start one another early, so a
 *   call may run beside any of them) -- for instance a sequence of
 *   attention calls over caches and queries that were all written earlier;
 * - calls that may overlap write distinct outputs, and every cache has its
 *   own workspace (the handle's epochs are per workspace).
 * That last non-overlapping launch has itself completed if it is one of
 * this library's: the kernels that write a cache (prefill, appends) let no
 * launch start before they complete, except a decode step's own attention,
 * and that attention lets later launches start only after its append has
 * completed.  The automatic split count changes with the setting (see
 * kivi_set_attention_splits), so results may differ in the last bits from
 * those of the setting off; with an explicit split count they are the same
 * bit for bit.  kivi_decode_step and kivi_decode_attention_static ignore
 * it.  Host only; no device work. */
kivi_status kivi_set_attention_overlap(kivi_cache *c, int enable);

/* Tokens held by every sequence; -2 when the sequences' lengths differ (see
 * kivi_cache_lengths), -1 if c is NULL. */
int kivi_cache_length(const kivi_cache *c);
kivi_status kivi_cache_reset(kivi_cache *c); /* length := 0; no device work */
void kivi_cache_destroy(kivi_cache *c);      /* NULL is a no-op */

const char *kivi_status_string(kivi_status s);
int kivi_last_cuda_error(void); /* cudaError_t of the last failed launch on this thread */

/* Diagnostics for the attention's failure path (no counterpart on the pages).
 * A packed split waits for each staged tile on an mbarrier, for at most
 * 200 ms; if a wait gives up, the split stops issuing copies, ORs 1 into the
 * workspace status word and still completes the merge protocol, so the
 * launch ends and the context stays usable.  An overlapping call (see
 * kivi_set_attention_overlap) waits, for at most 200 ms too, until the
 * previous call on its workspace has finished with a group's slots; if that
 * wait gives up it ORs 2 into the status word and goes on.  This call runs
 * the same bounded mbarrier wait in one CTA on a barrier phase that nothing
 * completes (no copy is issued and no thread arrives), then ORs 1 into
 * *status; then the same bounded epoch wait on an epoch that nothing
 * publishes, then ORs 2 into *status.
 * - status: one int, 4-byte aligned, device memory on the current device,
 *   or managed or mapped pinned host memory; the caller owns it and reads it
 *   after the stream has run the probe.
 * - Asynchronous on stream; the probe occupies one SM for about 400 ms.
 * - KIVI_EINVAL for a null, misaligned or unreachable pointer (nothing is
 *   launched); KIVI_ECUDA if the launch fails. */
kivi_status kivi_check_bounded_wait(int *status, void *stream);

/* Size of the library's fixed device scratch area used by
 * kivi_decode_attention_static: 8 MiB, held on every GPU that loads the
 * library until the process exits. */
#define KIVI_STATIC_WORKSPACE_BYTES (8u << 20)

/* Decode attention for callers that cannot allocate device memory where they
 * run it -- for example a plugin whose device memory must come from its host
 * framework's own pool, or a latency-critical path that cannot afford
 * cudaMalloc's implicit device-wide synchronization.  No counterpart on the
 * pages: it is kivi_decode_attention with the split-K scratch taken from the
 * library's own fixed device area (KIVI_STATIC_WORKSPACE_BYTES) instead of a
 * caller workspace.  Same q/out/scale contract and results as
 * kivi_decode_attention (bit for bit).
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * - Needs kivi_attention_workspace_bytes(c) <= KIVI_STATIC_WORKSPACE_BYTES,
 *   else KIVI_EWORKSPACE and nothing is launched.
 * - Runs on the calling thread's current device.  The first call on a device
 *   looks up the area's device address (cudaGetSymbolAddress) and caches it;
 *   make that first call before any stream capture.
 * - Each call clears the area's counters with one cudaMemsetAsync on stream.
 * - All calls share the one area and it keeps the last call's contents:
 *   calls that may overlap on the GPU (different streams, or different
 *   handles without ordering between them) race on it and must not be
 *   issued; serialize them on one stream.
 * - A staged-data wait that gives up (which only a device fault can cause)
 *   is recorded in the area's own status word, which no call reads back:
 *   use kivi_decode_attention with a workspace to observe it.
 * - Every argument check (device, pointers, lengths, size) is made before
 *   any CUDA call; a refused call does no device work. */
kivi_status kivi_decode_attention_static(kivi_cache *c, const void *q,
                                         kivi_dtype q_dtype, void *out,
                                         float softmax_scale, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_H */
