/*
 * kivi_oracle.c -- plain, slow, obviously correct CPU oracle of the KIVI
 * KV-cache hot path: the asymmetric min/max quantizer, the grouped + residual
 * cache (prefill and one-token append), and decode attention over the
 * dequantized cache.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
 * baseline of the benchmark; never by the product path.  No code is shared
 * with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (-ffp-contract=off matters: aarch64 gcc fuses a*b+c by default).
 *
 * Sources, by page (title, then section):
 *  [NB]  "KIVI - 2-bit KV cache quantisation" (llm-systems-cookbook, serving
 *        notebook 04), sections "Asymmetric 2-bit quantiser" and
 *        "K (per-channel) and V (per-token) quantisation".
 *  [VQ]  veloxquant-mlx docs, "KIVI", section "How it works" (items 1-4 and
 *        the zero/scale/q/recon formulas).
 *  [RV]  chooblog review "KIVI: A Tuning-Free Asymmetric 2bit Quantization for
 *        KV Cache (ICML'24)", §1.1 (quantization definition and worked
 *        example), §1.3 (decoding phase), §3.2.2-3.2.3 (grouped + residual
 *        split, Algorithm 1 prefill and decoding).
 *  [CQ]  "KV Cache Compression > Cache Quantization" (Brenndoerfer), the
 *        uniform quantization and dequantization formulas.
 *
 * Readings where the pages are silent or disagree:
 *  - every input element is first rounded to fp16 (the residual window is
 *    fp16 [VQ item 3]); codes are computed from those fp16 values widened;
 *  - round() is round-half-to-even (torch.round in [NB]);
 *  - the scale is stored as fp16 and the codes are computed with the stored
 *    fp16 scale, so decoding reproduces exactly what was encoded;
 *  - a zero range (or an fp16 scale that underflows to 0) stores scale 1
 *    ([NB] and [CQ] both replace a zero scale by one);
 *  - codes are clamped to [0, 2^b-1] ([NB] clamps);
 *  - default residual policy = [RV] Algorithm 1 read literally.
 */
#include "kivi_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE binary16 conversions, written from the format's definition:    */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals */
/* are f * 2^-24.  Rounding is to nearest, ties to even.               */
/* ------------------------------------------------------------------ */

float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  float v;
  if (e == 0)
    v = ldexpf((float)f, -24); /* zero or subnormal */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexpf((float)(f | 0x400), e - 25); /* 1.f * 2^(e-15) */
  return sign ? -v : v;
}

uint16_t orc_f32_to_f16(float x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7e00;
  double a = fabs((double)x);
  if (isinf(x)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  /* a = m * 2^k with m in [0.5, 1): the leading bit has weight 2^(k-1). */
  int k;
  frexp(a, &k);
  int lead = k - 1;                 /* exponent of the leading bit */
  int q_exp = lead < -14 ? -24 : lead - 10; /* weight of the last kept bit */
  double n = nearbyint(ldexp(a, -q_exp));   /* exact scaling, RNE */
  double v = ldexp(n, q_exp);               /* the rounded magnitude */
  if (v >= 65520.0) return sign | 0x7c00;   /* beyond max finite: inf */
  if (v < ldexp(1.0, -14)) {                /* subnormal (or rounded to 0) */
    return sign | (uint16_t)ldexp(v, 24);
  }
  frexp(v, &k);
  lead = k - 1;
  uint16_t frac = (uint16_t)(ldexp(v, 10 - lead) - 1024.0);
  return sign | (uint16_t)((lead + 15) << 10) | frac;
}

float orc_bf16_to_f32(uint16_t h) {
  /* bfloat16 is the upper half of a binary32 pattern. */
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round an input element of any accepted dtype to an fp16 bit pattern. */
static uint16_t ingest(const void *base, long idx, int dtype) {
  switch (dtype) {
  case ORC_F32:
    return orc_f32_to_f16(((const float *)base)[idx]);
  case ORC_F16:
    return ((const uint16_t *)base)[idx];
  default:
    return orc_f32_to_f16(orc_bf16_to_f32(((const uint16_t *)base)[idx]));
  }
}

/* ------------------------------------------------------------------ */
/* The quantizer ([VQ] "How it works"; [RV] §1.1; [NB] quantize_grouped):
 *   zero = min(group), scale = (max - min) / (2^b - 1),
 *   q = round((x - zero) / scale) clamped to [0, 2^b - 1],
 *   recon = q * scale + zero.                                          */
/* ------------------------------------------------------------------ */

void orc_quantize_group(const uint16_t *x, long n, long stride, int bits,
                        uint8_t *codes, long code_stride, uint16_t *scale16,
                        uint16_t *zero16, float *scale32) {
  const int L = (1 << bits) - 1;
  /* 1. min and max by a sequential scan */
  float mn = orc_f16_to_f32(x[0]);
  float mx = mn;
  for (long i = 1; i < n; i++) {
    float v = orc_f16_to_f32(x[i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  /* 2. range and fp32 scale (IEEE division) */
  float r = mx - mn;
  float s32 = r / (float)L;
  /* 3. stored fp16 scale; a zero range or an underflowed scale stores 1 */
  uint16_t sb = orc_f32_to_f16(s32);
  float s = orc_f16_to_f32(sb);
  if (r == 0.0f || s == 0.0f) {
    sb = 0x3c00; /* 1.0 */
    s = 1.0f;
  }
  /* 4. zero point = the minimum (an fp16 value already, so exact); -0 and
   *    +0 are the same minimum, and adding +0 stores it as +0 */
  uint16_t zb = orc_f32_to_f16(mn + 0.0f);
  float z = orc_f16_to_f32(zb);
  /* 5. codes: round half to even of (x - z) / s, then clamp */
  for (long i = 0; i < n; i++) {
    float v = orc_f16_to_f32(x[i * stride]);
    float d = v - z;
    float y = d / s;
    float q = rintf(y);
    if (q < 0.0f) q = 0.0f;
    if (q > (float)L) q = (float)L;
    codes[i * code_stride] = (uint8_t)q;
  }
  if (scale16) *scale16 = sb;
  if (zero16) *zero16 = zb;
  if (scale32) *scale32 = s32;
}

float orc_dequant(int q, uint16_t scale16, uint16_t zero16) {
  float p = (float)q * orc_f16_to_f32(scale16);
  return p + orc_f16_to_f32(zero16);
}

/* Packing (the pages fix no bit layout; this is the plain reading of "codes
 * packed to uint8"):
 * channel e of a row occupies bits [e*bits, e*bits + bits) of the row, LSB
 * first -- byte e*bits/8 at bit offset (e*bits) mod 8, a 3-bit code crossing
 * into the next byte when its offset is 6 or 7.  Keys and values, every
 * width, use this one layout. */
void orc_pack_row(const uint8_t *codes, int D, int bits, uint8_t *out) {
  if (D <= 0 || bits <= 0) return; /* an empty row packs to nothing */
  memset(out, 0, ((size_t)D * (size_t)bits + 7u) / 8u);
  for (int e = 0; e < D; e++)
    for (int j = 0; j < bits; j++) {
      const int bit = e * bits + j;
      out[bit / 8] |= (uint8_t)(((codes[e] >> j) & 1) << (bit % 8));
    }
}

void orc_unpack_row(const uint8_t *in, int D, int bits, uint8_t *codes) {
  for (int e = 0; e < D; e++) {
    int c = 0;
    for (int j = 0; j < bits; j++) {
      const int bit = e * bits + j;
      c |= ((in[bit / 8] >> (bit % 8)) & 1) << j;
    }
    codes[e] = (uint8_t)c;
  }
}

/* ------------------------------------------------------------------ */
/* Residual policy.
 * ALG1 ([RV] §3.2.2, Algorithm 1): K grouped part X_K[:l-r], r = l mod R;
 * V grouped part X_V[:l-R].
 * SHARED ([VQ] items 3-4): the newest R tokens stay fp16 for both K and V,
 * and aged-out tokens are quantized in whole multiples of G.            */
/* ------------------------------------------------------------------ */

long orc_nq_k(long l, int R, int G, int policy) {
  if (policy == ORC_POLICY_SHARED) {
    long a = l - R;
    return a > 0 ? (a / G) * G : 0;
  }
  return l - l % R;
}

long orc_nq_v(long l, int R, int G, int policy) {
  if (policy == ORC_POLICY_SHARED) return orc_nq_k(l, R, G, policy);
  return l > R ? l - R : 0;
}

/* Ring slots in the storage layout: R under ALG1 (the K residual is < R
 * tokens, the V residual <= R); R + G under SHARED (up to R + G - 1). */
static long ring_slots(int R, int G, int policy) {
  return policy == ORC_POLICY_SHARED ? (long)R + G : (long)R;
}

/* ------------------------------------------------------------------ */
/* The cache.  For clarity the oracle keeps the fp16 row of every token
 * it has seen (x16_k / x16_v); which rows count as "residual" follows
 * from the quantized counts alone.  Packed codes and fp16 scale/zero
 * are kept exactly in the storage layout.                             */
/* ------------------------------------------------------------------ */

struct orc_cache {
  int bits, G, R, D, B, H, policy;
  long Tcap, l;
  long nqk, nqv; /* tokens quantized so far (K, V) */
  int rowbytes;  /* D * bits / 8 */
  uint16_t *x16_k, *x16_v; /* [B][H][Tcap][D] */
  uint8_t *codes_k, *codes_v; /* [B][H][Tcap][rowbytes] */
  uint16_t *sk, *zk; /* [B][H][Tcap/G][D] */
  uint16_t *sv, *zv; /* [B][H][Tcap][D/G] */
  int n_out;         /* fp16 outlier key channels per key group (0: none) */
  uint8_t *oidx;     /* [B][H][Tcap/G][n_out] channels, largest first */
  uint16_t *oval;    /* [B][H][Tcap][n_out] their fp16 values */
};

orc_cache *orc_cache_new(int bits, int G, int R, int D, int B, int Hkv,
                         long Tcap, int policy) {
  if ((bits != 2 && bits != 3 && bits != 4 && bits != 8) || G <= 0 || R <= 0 ||
      D <= 0 || B <= 0 || Hkv <= 0 || Tcap <= 0)
    return NULL;
  if (D % G || R % G || Tcap % G || G % 4 || (D * bits) % 8) return NULL;
  orc_cache *c = (orc_cache *)calloc(1, sizeof *c);
  if (!c) return NULL;
  c->bits = bits;
  c->G = G;
  c->R = R;
  c->D = D;
  c->B = B;
  c->H = Hkv;
  c->Tcap = Tcap;
  c->policy = policy;
  c->rowbytes = D * bits / 8;
  size_t units = (size_t)B * Hkv;
  c->x16_k = calloc(units * Tcap * D, sizeof(uint16_t));
  c->x16_v = calloc(units * Tcap * D, sizeof(uint16_t));
  c->codes_k = calloc(units * Tcap * c->rowbytes, 1);
  c->codes_v = calloc(units * Tcap * c->rowbytes, 1);
  c->sk = calloc(units * (Tcap / G) * D, sizeof(uint16_t));
  c->zk = calloc(units * (Tcap / G) * D, sizeof(uint16_t));
  c->sv = calloc(units * Tcap * (D / G), sizeof(uint16_t));
  c->zv = calloc(units * Tcap * (D / G), sizeof(uint16_t));
  if (!c->x16_k || !c->x16_v || !c->codes_k || !c->codes_v || !c->sk ||
      !c->zk || !c->sv || !c->zv) {
    orc_cache_free(c);
    return NULL;
  }
  return c;
}

void orc_cache_free(orc_cache *c) {
  if (!c) return;
  free(c->x16_k);
  free(c->x16_v);
  free(c->codes_k);
  free(c->codes_v);
  free(c->sk);
  free(c->zk);
  free(c->sv);
  free(c->zv);
  free(c->oidx);
  free(c->oval);
  free(c);
}

/* Outlier-aware keys ([NB] Exercises, item 2: keep the top-1% of K channels
 * at fp16 and quantise the rest).  Reading: per key group (G tokens; every
 * channel is its own quantization group), the n_out channels with the
 * largest max |x| over the group's tokens are kept as fp16 values, chosen
 * largest first, ties to the lower channel.  Their codes, scales and zeros
 * are stored as 0, so the packed group decodes to 0 on them, and the decoded
 * key takes the kept value.  The other channels are quantized as without
 * outliers.  On an empty cache only; n_out in [0, 8]. */
int orc_cache_set_outliers(orc_cache *c, int n_out) {
  if (c->l != 0 || n_out < 0 || n_out > 8 || n_out > c->D) return -1;
  free(c->oidx);
  free(c->oval);
  c->oidx = NULL;
  c->oval = NULL;
  c->n_out = n_out;
  if (n_out == 0) return 0;
  size_t units = (size_t)c->B * c->H;
  c->oidx = calloc(units * (c->Tcap / c->G) * n_out, 1);
  c->oval = calloc(units * c->Tcap * n_out, sizeof(uint16_t));
  return c->oidx && c->oval ? 0 : -1;
}

int orc_cache_outliers(const orc_cache *c) { return c->n_out; }

long orc_cache_length(const orc_cache *c) { return c->l; }

static size_t unit_of(const orc_cache *c, int b, int h) {
  return (size_t)b * c->H + h;
}

/* Per-channel K quantization of one group: tokens t0..t0+G-1 of (b, h).
 * Each channel d is one group of G tokens ([VQ] item 1, [NB] K along
 * dim 0 with group 32). */
static void quantize_k_group(orc_cache *c, int b, int h, long t0) {
  const int D = c->D, G = c->G;
  size_t u = unit_of(c, b, h);
  const uint16_t *x = c->x16_k + (u * c->Tcap + t0) * D;
  uint8_t *codes = (uint8_t *)malloc((size_t)G * D);
  long g = t0 / G;
  for (int d = 0; d < D; d++) {
    orc_quantize_group(x + d, G, D, c->bits, codes + d, D,
                       &c->sk[(u * (c->Tcap / G) + g) * D + d],
                       &c->zk[(u * (c->Tcap / G) + g) * D + d], NULL);
  }
  if (c->n_out > 0) {
    float *amax = (float *)malloc((size_t)D * sizeof(float));
    char *chosen = (char *)calloc((size_t)D, 1);
    for (int d = 0; d < D; d++) {
      float m = 0.0f;
      for (int i = 0; i < G; i++) {
        float a = fabsf(orc_f16_to_f32(x[(size_t)i * D + d]));
        if (a > m) m = a;
      }
      amax[d] = m;
    }
    for (int o = 0; o < c->n_out; o++) {
      int best = -1;
      for (int d = 0; d < D; d++)
        if (!chosen[d] && (best < 0 || amax[d] > amax[best])) best = d;
      chosen[best] = 1;
      c->oidx[(u * (c->Tcap / G) + g) * c->n_out + o] = (uint8_t)best;
      c->sk[(u * (c->Tcap / G) + g) * D + best] = 0;
      c->zk[(u * (c->Tcap / G) + g) * D + best] = 0;
      for (int i = 0; i < G; i++) {
        codes[(size_t)i * D + best] = 0;
        c->oval[(u * c->Tcap + t0 + i) * c->n_out + o] = x[(size_t)i * D + best];
      }
    }
    free(amax);
    free(chosen);
  }
  for (int i = 0; i < G; i++)
    orc_pack_row(codes + (size_t)i * D, D, c->bits, c->codes_k + (u * c->Tcap + t0 + i) * c->rowbytes);
  free(codes);
}

/* Per-token V quantization of token t of (b, h): D/G groups of G
 * consecutive channels ([VQ] item 2; [RV] Step C, numGroup = d // G). */
static void quantize_v_token(orc_cache *c, int b, int h, long t) {
  const int D = c->D, G = c->G;
  size_t u = unit_of(c, b, h);
  const uint16_t *x = c->x16_v + (u * c->Tcap + t) * D;
  uint8_t codes[4096];
  for (int gg = 0; gg < D / G; gg++) {
    orc_quantize_group(x + gg * G, G, 1, c->bits, codes + gg * G, 1,
                       &c->sv[(u * c->Tcap + t) * (D / G) + gg],
                       &c->zv[(u * c->Tcap + t) * (D / G) + gg], NULL);
  }
  orc_pack_row(codes, D, c->bits, c->codes_v + (u * c->Tcap + t) * c->rowbytes);
}

/* Bring the quantized parts up to the policy's counts for length l.
 * K is quantized in whole groups of G tokens; V token by token. */
static void advance_quantized(orc_cache *c, long l) {
  long want_k = orc_nq_k(l, c->R, c->G, c->policy);
  long want_v = orc_nq_v(l, c->R, c->G, c->policy);
  for (int b = 0; b < c->B; b++)
    for (int h = 0; h < c->H; h++) {
      for (long t0 = c->nqk; t0 < want_k; t0 += c->G) quantize_k_group(c, b, h, t0);
      for (long t = c->nqv; t < want_v; t++) quantize_v_token(c, b, h, t);
    }
  c->nqk = want_k;
  c->nqv = want_v;
}

/* Prefill ([RV] Algorithm 1, prefill steps B-D): the whole prompt arrives at
 * once; the grouped parts are quantized, the rest stays fp16. */
int orc_cache_prefill(orc_cache *c, const void *k, const void *v, int dtype,
                      long T) {
  if (c->l != 0 || T < 0 || T > c->Tcap) return -1;
  const int D = c->D;
  for (int b = 0; b < c->B; b++)
    for (int h = 0; h < c->H; h++) {
      size_t u = unit_of(c, b, h);
      for (long t = 0; t < T; t++)
        for (int d = 0; d < D; d++) {
          long src = ((long)u * T + t) * D + d;
          c->x16_k[(u * c->Tcap + t) * D + d] = ingest(k, src, dtype);
          c->x16_v[(u * c->Tcap + t) * D + d] = ingest(v, src, dtype);
        }
    }
  advance_quantized(c, T);
  c->l = T;
  return 0;
}

/* Decode-time append ([RV] §1.3 step 1, concat; §3.2.3 decoding phase):
 * when the K residual reaches R it is quantized whole and emptied; when the
 * V residual exceeds R its oldest token is quantized. */
int orc_cache_append(orc_cache *c, const void *k1, const void *v1, int dtype) {
  if (c->l >= c->Tcap) return -1;
  const int D = c->D;
  long t = c->l;
  for (int b = 0; b < c->B; b++)
    for (int h = 0; h < c->H; h++) {
      size_t u = unit_of(c, b, h);
      for (int d = 0; d < D; d++) {
        long src = (long)u * D + d;
        c->x16_k[(u * c->Tcap + t) * D + d] = ingest(k1, src, dtype);
        c->x16_v[(u * c->Tcap + t) * D + d] = ingest(v1, src, dtype);
      }
    }
  advance_quantized(c, t + 1);
  c->l = t + 1;
  return 0;
}

void orc_cache_export(const orc_cache *c, uint8_t *codes_k, uint16_t *scale_k,
                      uint16_t *zero_k, uint8_t *codes_v, uint16_t *scale_v,
                      uint16_t *zero_v, uint16_t *ring_k, uint16_t *ring_v) {
  const int D = c->D, G = c->G;
  const long W = ring_slots(c->R, c->G, c->policy);
  const size_t units = (size_t)c->B * c->H;
  if (codes_k) memset(codes_k, 0, units * c->Tcap * c->rowbytes);
  if (codes_v) memset(codes_v, 0, units * c->Tcap * c->rowbytes);
  if (scale_k) memset(scale_k, 0, units * (c->Tcap / G) * D * 2);
  if (zero_k) memset(zero_k, 0, units * (c->Tcap / G) * D * 2);
  if (scale_v) memset(scale_v, 0, units * c->Tcap * (D / G) * 2);
  if (zero_v) memset(zero_v, 0, units * c->Tcap * (D / G) * 2);
  if (ring_k) memset(ring_k, 0, units * W * D * 2);
  if (ring_v) memset(ring_v, 0, units * W * D * 2);
  for (size_t u = 0; u < units; u++) {
    if (codes_k)
      memcpy(codes_k + u * c->Tcap * c->rowbytes,
             c->codes_k + u * c->Tcap * c->rowbytes, (size_t)c->nqk * c->rowbytes);
    if (codes_v)
      memcpy(codes_v + u * c->Tcap * c->rowbytes,
             c->codes_v + u * c->Tcap * c->rowbytes, (size_t)c->nqv * c->rowbytes);
    if (scale_k)
      memcpy(scale_k + u * (c->Tcap / G) * D, c->sk + u * (c->Tcap / G) * D,
             (size_t)(c->nqk / G) * D * 2);
    if (zero_k)
      memcpy(zero_k + u * (c->Tcap / G) * D, c->zk + u * (c->Tcap / G) * D,
             (size_t)(c->nqk / G) * D * 2);
    if (scale_v)
      memcpy(scale_v + u * c->Tcap * (D / G), c->sv + u * c->Tcap * (D / G),
             (size_t)c->nqv * (D / G) * 2);
    if (zero_v)
      memcpy(zero_v + u * c->Tcap * (D / G), c->zv + u * c->Tcap * (D / G),
             (size_t)c->nqv * (D / G) * 2);
    for (long t = c->nqk; t < c->l; t++)
      if (ring_k)
        memcpy(ring_k + (u * W + t % W) * D, c->x16_k + (u * c->Tcap + t) * D,
               (size_t)D * 2);
    for (long t = c->nqv; t < c->l; t++)
      if (ring_v)
        memcpy(ring_v + (u * W + t % W) * D, c->x16_v + (u * c->Tcap + t) * D,
               (size_t)D * 2);
  }
}

/* The outlier channels and values of the quantized key groups / rows
 * (zeros elsewhere): idx [B][H][Tcap/G][n_out], val [B][H][Tcap][n_out]. */
void orc_cache_export_outliers(const orc_cache *c, uint8_t *idx, uint16_t *val) {
  const int G = c->G, n = c->n_out;
  const size_t units = (size_t)c->B * c->H;
  if (n == 0) return;
  memset(idx, 0, units * (c->Tcap / G) * n);
  memset(val, 0, units * c->Tcap * n * 2);
  for (size_t u = 0; u < units; u++) {
    memcpy(idx + u * (c->Tcap / G) * n, c->oidx + u * (c->Tcap / G) * n, (size_t)(c->nqk / G) * n);
    memcpy(val + u * c->Tcap * n, c->oval + u * c->Tcap * n, (size_t)c->nqk * n * 2);
  }
}

/* K-hat and V-hat of one (b, h): quantized rows decoded from the packed
 * bytes ([VQ] recon = q * scale + zero), residual rows widened from fp16. */
void orc_cache_dequant(const orc_cache *c, int b, int h, float *khat,
                       float *vhat) {
  const int D = c->D, G = c->G;
  size_t u = unit_of(c, b, h);
  uint8_t codes[4096];
  for (long t = 0; t < c->l; t++) {
    if (t < c->nqk) {
      orc_unpack_row(c->codes_k + (u * c->Tcap + t) * c->rowbytes, D, c->bits, codes);
      long g = t / G;
      for (int d = 0; d < D; d++)
        khat[t * D + d] =
            orc_dequant(codes[d], c->sk[(u * (c->Tcap / G) + g) * D + d],
                        c->zk[(u * (c->Tcap / G) + g) * D + d]);
      for (int o = 0; o < c->n_out; o++)
        khat[t * D + c->oidx[(u * (c->Tcap / G) + g) * c->n_out + o]] =
            orc_f16_to_f32(c->oval[(u * c->Tcap + t) * c->n_out + o]);
    } else {
      for (int d = 0; d < D; d++)
        khat[t * D + d] = orc_f16_to_f32(c->x16_k[(u * c->Tcap + t) * D + d]);
    }
    if (t < c->nqv) {
      orc_unpack_row(c->codes_v + (u * c->Tcap + t) * c->rowbytes, D, c->bits, codes);
      for (int d = 0; d < D; d++)
        vhat[t * D + d] =
            orc_dequant(codes[d], c->sv[(u * c->Tcap + t) * (D / G) + d / G],
                        c->zv[(u * c->Tcap + t) * (D / G) + d / G]);
    } else {
      for (int d = 0; d < D; d++)
        vhat[t * D + d] = orc_f16_to_f32(c->x16_v[(u * c->Tcap + t) * D + d]);
    }
  }
}

/* Decode attention ([RV] §1.3 step 2: A = softmax(t_Q X_K^T), t_O = A X_V;
 * [NB] attn(): scores scaled by 1/sqrt(D)).  fp32, fixed order:
 * score_t = (sum_d q_d * khat_td, d ascending) * scale; m = max_t score_t;
 * e_t = expf(score_t - m); l = sum_t e_t (t ascending);
 * out_d = (sum_t e_t * vhat_td, t ascending) / l. */
int orc_decode_attention(const orc_cache *c, const float *q, int Hq,
                         float scale, float *out) {
  const int D = c->D;
  const long l = c->l;
  if (l <= 0 || Hq <= 0 || Hq % c->H) return -1;
  const int grp = Hq / c->H;
  if (scale <= 0.0f) scale = 1.0f / sqrtf((float)D);
  float *khat = (float *)malloc((size_t)l * D * sizeof(float));
  float *vhat = (float *)malloc((size_t)l * D * sizeof(float));
  float *e = (float *)malloc((size_t)l * sizeof(float));
  if (!khat || !vhat || !e) {
    free(khat);
    free(vhat);
    free(e);
    return -1;
  }
  for (int b = 0; b < c->B; b++)
    for (int h = 0; h < c->H; h++) {
      orc_cache_dequant(c, b, h, khat, vhat);
      for (int jj = 0; jj < grp; jj++) {
        int j = h * grp + jj;
        const float *qv = q + ((size_t)b * Hq + j) * D;
        float *o = out + ((size_t)b * Hq + j) * D;
        float m = -INFINITY;
        for (long t = 0; t < l; t++) {
          float acc = 0.0f;
          for (int d = 0; d < D; d++) acc += qv[d] * khat[t * D + d];
          e[t] = acc * scale;
          if (e[t] > m) m = e[t];
        }
        float den = 0.0f;
        for (long t = 0; t < l; t++) {
          e[t] = expf(e[t] - m);
          den += e[t];
        }
        for (int d = 0; d < D; d++) {
          float num = 0.0f;
          for (long t = 0; t < l; t++) num += e[t] * vhat[t * D + d];
          o[d] = num / den;
        }
      }
    }
  free(khat);
  free(vhat);
  free(e);
  return 0;
}

void orc_attention_f64(const float *q, const float *k, const float *v, long l,
                       int D, double scale, double *out) {
  double *s = (double *)malloc((size_t)l * sizeof(double));
  double m = -INFINITY, den = 0.0;
  for (long t = 0; t < l; t++) {
    double acc = 0.0;
    for (int d = 0; d < D; d++) acc += (double)q[d] * (double)k[t * D + d];
    s[t] = acc * scale;
    if (s[t] > m) m = s[t];
  }
  for (long t = 0; t < l; t++) {
    s[t] = exp(s[t] - m);
    den += s[t];
  }
  for (int d = 0; d < D; d++) {
    double num = 0.0;
    for (long t = 0; t < l; t++) num += s[t] * (double)v[t * D + d];
    out[d] = num / den;
  }
  free(s);
}
