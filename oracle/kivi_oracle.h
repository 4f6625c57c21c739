/*
 * kivi_oracle.h -- the slow, plain CPU oracle for the KIVI KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; both sides are written
 * independently from the pages that describe the method.
 *
 * Precision: the quantizer and the reference attention run in fp32 with a
 * fixed, sequential operation order (the notebook "KIVI - 2-bit KV cache
 * quantisation" computes everything after `x.float()`), compiled with
 * -ffp-contract=off so that no multiply-add is fused.  A double-precision
 * brute-force attention is provided for tiny inputs.
 *
 * Storage layout of the oracle's cache (the plain reading; the pages fix no
 * packing):
 *   codes_k [B][Hkv][Tcap][D*bits/8]   token-major packed rows
 *   scale_k, zero_k [B][Hkv][Tcap/G][D] fp16 bit patterns
 *   codes_v [B][Hkv][Tcap][D*bits/8]
 *   scale_v, zero_v [B][Hkv][Tcap][D/G] fp16 bit patterns
 *   ring_k, ring_v  [B][Hkv][R][D]      fp16, token t in slot t mod R
 * Channel e of a packed row (keys and values, every width) occupies bits
 * [e*bits, e*bits + bits), LSB first: byte (e*bits)/8 at bit (e*bits)%8, a
 * 3-bit code crossing into the next byte when that offset is 6 or 7.
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Input element types accepted by prefill / append. */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* Residual policies. */
enum {
  ORC_POLICY_ALG1 = 0,   /* KIVI review, Algorithm 1: K residual = l mod R, V residual = R */
  ORC_POLICY_SHARED = 1  /* VeloxQuant reading: both keep >= R fp16 tokens, shared G-aligned edge */
};

/* IEEE binary16 <-> binary32, round to nearest even. */
uint16_t orc_f32_to_f16(float x);
float orc_f16_to_f32(uint16_t h);
float orc_bf16_to_f32(uint16_t h);

/* One quantization group (the min/max quantizer of every page).
 * x: n fp16 bit patterns, element i at x[i*stride].
 * Writes n codes (unpacked, one per byte) to codes[i*code_stride],
 * the stored fp16 scale and zero, and the fp32 scale before rounding. */
void orc_quantize_group(const uint16_t *x, long n, long stride, int bits,
                        uint8_t *codes, long code_stride,
                        uint16_t *scale16, uint16_t *zero16, float *scale32);

/* Dequantize one code: fl(fl(q*s) + z), no fused multiply-add. */
float orc_dequant(int q, uint16_t scale16, uint16_t zero16);

/* Pack / unpack a row of D codes (LSB-first, channel e at bits
 * [e*bits, e*bits + bits) of the row). */
void orc_pack_row(const uint8_t *codes, int D, int bits, uint8_t *out);
void orc_unpack_row(const uint8_t *in, int D, int bits, uint8_t *codes);

/* Token counts held quantized after l tokens under a policy. */
long orc_nq_k(long l, int R, int G, int policy);
long orc_nq_v(long l, int R, int G, int policy);

/* ---- the cache ---- */
typedef struct orc_cache orc_cache;

orc_cache *orc_cache_new(int bits, int G, int R, int D, int B, int Hkv,
                         long Tcap, int policy);
void orc_cache_free(orc_cache *c);
long orc_cache_length(const orc_cache *c);

/* Prefill an empty cache with T tokens; k, v are [B][Hkv][T][D] of dtype.
 * Returns 0, or -1 on a bad state/shape. */
int orc_cache_prefill(orc_cache *c, const void *k, const void *v, int dtype,
                      long T);
/* Append one token; k1, v1 are [B][Hkv][D]. Returns 0 or -1. */
int orc_cache_append(orc_cache *c, const void *k1, const void *v1, int dtype);

/* Copy the cache state out in the storage layout above.  Any pointer may be
 * NULL.  Rows/slots that hold no live token are written as zero. */
/* Outlier-aware keys (fp16 outlier channels per key group); see the .c. */
int orc_cache_set_outliers(orc_cache *c, int n_out);
int orc_cache_outliers(const orc_cache *c);
void orc_cache_export_outliers(const orc_cache *c, uint8_t *idx, uint16_t *val);

void orc_cache_export(const orc_cache *c, uint8_t *codes_k, uint16_t *scale_k,
                      uint16_t *zero_k, uint8_t *codes_v, uint16_t *scale_v,
                      uint16_t *zero_v, uint16_t *ring_k, uint16_t *ring_v);

/* Dequantized K-hat and V-hat of one (b, kv-head): [l][D] fp32 each.
 * Packed rows are unpacked from the packed bytes; residual rows are the fp16
 * values widened. */
void orc_cache_dequant(const orc_cache *c, int b, int h, float *khat,
                       float *vhat);

/* Decode attention over the cache, fp32, fixed order.
 * q: [B][Hq][D] fp32; out: [B][Hq][D] fp32; scale <= 0 means 1/sqrt(D).
 * Query head j reads KV head j / (Hq/Hkv). Returns 0 or -1. */
int orc_decode_attention(const orc_cache *c, const float *q, int Hq,
                         float scale, float *out);

/* Brute-force attention in double for one query over explicit K, V rows:
 * k, v: [l][D] fp32, q: [D] fp32, out: [D] double. */
void orc_attention_f64(const float *q, const float *k, const float *v, long l,
                       int D, double scale, double *out);

#ifdef __cplusplus
}
#endif
#endif
