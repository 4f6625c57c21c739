// quantize.cu -- prefill quantize/pack and decode append/flush kernels.
//
// Grouping (veloxquant-mlx "KIVI", How it works items 1-2; notebook "KIVI -
// 2-bit KV cache quantisation", K along dim 0 and V along dim 1 with group
// 32): keys per channel over groups of G = 32 tokens, values per token over
// groups of G = 32 channels.  Residual split (chooblog KIVI review, §3.2.2
// and Algorithm 1): the first nq_k = R*floor(l/R) keys and nq_v = max(l-R, 0)
// values are quantized, the rest stay fp16 in a ring of R slots.
#include <climits>

#include "quant_common.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Value rows are group-interleaved: the unit of 4 channels 32*gp + 4*w .. +3
// (bits/2 bytes) is stored at unit position 4*w + gp.
__device__ __forceinline__ int v_unit_pos(int unit) { return 4 * (unit & 7) + (unit >> 3); }


// ---------------------------------------------------------------------------
// Prefill quantizer arithmetic.
//
// The code of x is rint(fl(fl(x - z) / s)) with the stored fp16 scale s.  The
// IEEE quotient is obtained without a division instruction by one residual
// correction of a reciprocal estimate (Markstein's refinement of a quotient):
// with d = fl(x - z), inv ~ 1/s (rcp.approx, relative error below 2^-22) and
// y1 = fl(d * inv), the residual r = fma(-y1, s, d) is exact (d - y1*s has at
// most 13 significant bits), and y2 = fma(r, inv, y1) is the rounding of a
// value within 2^-44 (relative) of d / s.  d has 24 significant bits and s
// 11, so d / s is never a rounding midpoint of fp32 and lies at least 2^-35
// (relative) away from every midpoint; hence y2 = fl(d / s) exactly.  When s
// is an fp16 normal number, y2 < L + 1/2 (s differs from (max - min)/L by at
// most 2^-11 relative), so no clamp is needed; groups whose stored scale is an
// fp16 subnormal use the IEEE division and the clamp.
//
// rint(y2) is read off t = y2 + 1.5 * 2^23, whose bit pattern is
// 0x4B400000 + rint(y2); the codes of a word are summed as t_bits << shift
// (mod 2^32) and the constant sum of the 0x4B400000 << shift terms removed.

struct FastParams {
  float inv;
  bool safe;
};

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ FastParams fast_params(const GroupParams& p) {
  FastParams f;
  f.inv = rcp_approx(p.s);
  f.safe = p.s >= 6.103515625e-05f;  // fp16 normal
  return f;
}

__device__ __forceinline__ uint32_t code_bits(float x, float z, float s, float inv) {
  const float d = __fsub_rn(x, z);
  const float y1 = __fmul_rn(d, inv);
  const float r = fmaf(-y1, s, d);
  const float y2 = fmaf(r, inv, y1);
  return __float_as_uint(__fadd_rn(y2, kRoundMagic));
}

// sum over e < n of (0x4B400000 << (bits * e)) mod 2^32
__host__ __device__ constexpr uint32_t magic_sum(int n, int bits) {
  uint32_t c = 0;
  for (int e = 0; e < n; ++e) c += kRoundMagicBits << (bits * e);
  return c;
}

__device__ __forceinline__ uint32_t exact_code(float x, float z, float s, int L) {
  const int q = __float2int_rn(__fdiv_rn(__fsub_rn(x, z), s));
  return (uint32_t)min(max(q, 0), L);
}

// Exact codes of 8 key channels of one token (each channel its own group),
// packed LSB-first: 8 * BITS bits, as two words (the second one used at 8
// bits only).
template <int BITS>
__device__ __noinline__ uint2 exact_key_slice(uint4 xb, const float* z, const float* s) {
  constexpr int L = (1 << BITS) - 1;
  const uint32_t w[4] = {xb.x, xb.y, xb.z, xb.w};
  uint32_t acc[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float x = __half2float(__ushort_as_half((unsigned short)(w[e >> 1] >> (16 * (e & 1)))));
    const int bit = BITS * e;
    acc[bit >> 5] |= exact_code(x, z[e], s[e], L) << (bit & 31);
  }
  return make_uint2(acc[0], acc[1]);
}

// Store this lane's 8 key codes (8 * BITS bits) at dst.
template <int BITS>
__device__ __forceinline__ void store_key_slice(uint8_t* dst, uint2 acc) {
  if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)acc.x;
  else if constexpr (BITS == 4) *reinterpret_cast<uint32_t*>(dst) = acc.x;
  else *reinterpret_cast<uint2*>(dst) = acc;
}

// Exact codes of one value group (32 channels, one scale/zero).
template <int BITS>
__device__ __noinline__ void exact_value_group(const uint32_t* xw, float z, float s,
                                               uint32_t* words) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int CPW = 32 / BITS;  // codes per word
#pragma unroll
  for (int w = 0; w < BITS; ++w) words[w] = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x = __half2float(__ushort_as_half((unsigned short)(xw[e >> 1] >> (16 * (e & 1)))));
    words[e / CPW] |= exact_code(x, z, s, L) << (BITS * (e % CPW));
  }
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) {
  return (uint32_t)__half_as_ushort(__low2half(v)) | ((uint32_t)__half_as_ushort(__high2half(v)) << 16);
}

__device__ __forceinline__ uint32_t pack_halves(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// Element e (0..7) of 8 halves held as 4 half2, without dynamic register
// indexing.
__device__ __forceinline__ __half pick_half(const __half2 (&v)[4], int e) {
  __half2 p = v[0];
  p = (e >> 1) == 1 ? v[1] : p;
  p = (e >> 1) == 2 ? v[2] : p;
  p = (e >> 1) == 3 ? v[3] : p;
  return (e & 1) ? __high2half(p) : __low2half(p);
}

__device__ __forceinline__ uint4 h2x4_bits(const __half2 (&v)[4]) {
  return make_uint4(h2_bits(v[0]), h2_bits(v[1]), h2_bits(v[2]), h2_bits(v[3]));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem));
}

// 8 consecutive input elements staged in shared memory -> fp16 (nearest even).
template <int DT>
__device__ __forceinline__ void smem8(const uint4* p, __half2 (&h)[4]);

template <>
__device__ __forceinline__ void smem8<kF16>(const uint4* p, __half2 (&h)[4]) {
  const uint4 u = *p;
  h[0] = *reinterpret_cast<const __half2*>(&u.x);
  h[1] = *reinterpret_cast<const __half2*>(&u.y);
  h[2] = *reinterpret_cast<const __half2*>(&u.z);
  h[3] = *reinterpret_cast<const __half2*>(&u.w);
}

template <>
__device__ __forceinline__ void smem8<kBF16>(const uint4* p, __half2 (&h)[4]) {
  const uint4 u = *p;
  h[0] = bf16x2_to_half2(u.x);
  h[1] = bf16x2_to_half2(u.y);
  h[2] = bf16x2_to_half2(u.z);
  h[3] = bf16x2_to_half2(u.w);
}

template <>
__device__ __forceinline__ void smem8<kF32>(const uint4* p, __half2 (&h)[4]) {
  const uint4 a = p[0], b = p[1];
  h[0] = __floats2half2_rn(__uint_as_float(a.x), __uint_as_float(a.y));
  h[1] = __floats2half2_rn(__uint_as_float(a.z), __uint_as_float(a.w));
  h[2] = __floats2half2_rn(__uint_as_float(b.x), __uint_as_float(b.y));
  h[3] = __floats2half2_rn(__uint_as_float(b.z), __uint_as_float(b.w));
}

// Store the 8 packed units of value group g (channels 32g + 4u .. +3) of one
// row at their interleaved positions 4u + g.
template <int BITS>
__device__ __forceinline__ void store_value_units(uint8_t* row, int g, const uint32_t (&words)[BITS]) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if constexpr (BITS == 2)
      row[v_unit_pos(8 * g + u)] = (uint8_t)(words[u >> 2] >> (8 * (u & 3)));
    else if constexpr (BITS == 4)
      reinterpret_cast<uint16_t*>(row)[v_unit_pos(8 * g + u)] = (uint16_t)(words[u >> 1] >> (16 * (u & 1)));
    else
      reinterpret_cast<uint32_t*>(row)[v_unit_pos(8 * g + u)] = words[u];
  }
}

// One CTA = one 32-token chunk of one (b, kv-head): warp 0 quantizes the
// chunk's keys (one K group per channel: 128 channels x 32 tokens), warp 1
// its values (32 tokens x 4 channel groups).  Each warp first stages its raw
// 32-row input tile in shared memory with cp.async (rows 16-byte chunked;
// the value tile's chunks XOR-swizzled so that the group reads below are
// bank-conflict free), then:
//   keys:   lane l owns channels 8*(l%16) .. +7 of the rows of parity l/16;
//           the two parities' min/max meet in one shuffle;
//   values: lane l owns, in round rr, the whole 32-channel group l%4 of row
//           8*rr + l/4, so min, max and the scale are computed once per group.
// Value-tile swizzle (16-bit inputs): chunk j of group g of row r sits at
// 4g + (j ^ ((g >> 1) | ((r & 1) << 1))), so the 8 lanes of a shared-memory
// phase (rows r, r+1; groups 0..3) hit distinct 16-byte bank slots.  fp32 rows
// (two chunks per 8 elements, CPG = 8) are left unswizzled.
template <int CPG>
__device__ __forceinline__ int vswz(int r, int c) {
  if constexpr (CPG != 4) {
    return c;
  } else {
    const int g = c >> 2, j = c & 3;
    return 4 * g + (j ^ ((g >> 1) | ((r & 1) << 1)));
  }
}

// Quantizes this warp's half of one staged 32-token chunk t0 = 32 * chunk:
// the keys for warp 0, the values for warp 1.  kq: quantize the chunk's key
// group (one per channel); key rows t >= kring (t < T) go to the ring as
// fp16.  Value rows t in [vlo, vhi) are quantized (one group per 32
// channels); value rows t >= vring outside that range (t < T) go to the ring.
// s_in holds the chunk's input rows in the layout of DT (value rows
// swizzled by vswz).
//   keys:   lane l owns channels 8*(l%16) .. +7 of the rows of parity l/16;
//           the two parities' min/max meet in one shuffle;
//   values: lane l owns, in round rr, the whole 32-channel group l%4 of row
//           8*rr + l/4, so min, max and the scale are computed once per group.
template <int BITS, int DT, bool OUTL>
__device__ __forceinline__ void quantize_chunk(const CacheView& cv, const uint4* s_in, uint8_t* s_codes,
                                               long unit, int chunk, int T, bool kq, int kring, int vlo,
                                               int vhi, int vring) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;          // packed bytes per token row
  constexpr int EB = DT == kF32 ? 4 : 2;           // input bytes per element
  constexpr int CPR = kHeadDim * EB / 16;          // 16-byte chunks per input row
  constexpr int CPG = CPR / 4;                     // chunks per 32-channel group
  constexpr int CPE = EB / 2;                      // chunks per 8 elements
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = chunk * 32;

  if (warp == 0) {
    // ---------------- keys ----------------
    const int cl = lane & 15, par = lane >> 4;
    const int c8 = cl * 8;
    if (kq) {
      __half2 mn[4], mx[4], x[4];
      smem8<DT>(&s_in[par * CPR + cl * CPE], x);
#pragma unroll
      for (int i = 0; i < 4; ++i) mn[i] = mx[i] = x[i];
#pragma unroll
      for (int k = 1; k < 16; ++k) {
        smem8<DT>(&s_in[(2 * k + par) * CPR + cl * CPE], x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mn[i] = __hmin2(mn[i], x[i]);
          mx[i] = __hmax2(mx[i], x[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // the other token parity
        mn[i] = __hmin2(mn[i], __shfl_xor_sync(kFull, mn[i], 16));
        mx[i] = __hmax2(mx[i], __shfl_xor_sync(kFull, mx[i], 16));
      }
      GroupParams gp[8];
      float inv[8], zf[8], sf[8];
      bool safe = true;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        gp[2 * i] = group_params(__low2float(mn[i]), __low2float(mx[i]), L);
        gp[2 * i + 1] = group_params(__high2float(mn[i]), __high2float(mx[i]), L);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const FastParams f = fast_params(gp[e]);
        inv[e] = f.inv;
        zf[e] = gp[e].z;
        sf[e] = gp[e].s;
        safe = safe && f.safe;
      }
      // codes per 32-bit word, and the correction of a word's magic sum
      constexpr int CW = BITS == 8 ? 4 : 8;
      constexpr uint32_t C = magic_sum(CW, BITS);
      // Outlier-aware keys: the n_out channels of the group with the largest
      // max |k| (largest first, ties to the lower channel) stay fp16; their
      // codes, scales and zeros become 0.  Every lane takes part in each
      // round's argmax (the two token parities hold the same channels).
      int och[kMaxOutliers] = {0, 0, 0, 0};
      uint32_t keep0 = ~0u, keep1 = ~0u;  // code bits of this lane's kept (non-outlier) channels
      uint32_t keepm = 0xffu;             // bit e: channel c8 + e is kept
      if constexpr (OUTL) {
        float am[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          am[2 * i] = fmaxf(fabsf(__low2float(mn[i])), fabsf(__low2float(mx[i])));
          am[2 * i + 1] = fmaxf(fabsf(__high2float(mn[i])), fabsf(__high2float(mx[i])));
        }
        uint32_t mine = 0;  // bit e: channel c8 + e is an outlier
#pragma unroll
        for (int o = 0; o < kMaxOutliers; ++o) {
          if (o < cv.n_out) {
            float bv = -1.0f;
            int bc = 0x7fffffff;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (!((mine >> e) & 1u) && am[e] > bv) {
                bv = am[e];
                bc = c8 + e;
              }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
              const float ov = __shfl_xor_sync(kFull, bv, off);
              const int oc = __shfl_xor_sync(kFull, bc, off);
              if (ov > bv || (ov == bv && oc < bc)) {
                bv = ov;
                bc = oc;
              }
            }
            och[o] = bc;
            if ((bc >> 3) == cl) mine |= 1u << (bc & 7);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if ((mine >> e) & 1u) {
            gp[e].sh = __ushort_as_half((unsigned short)0);
            gp[e].zh = __ushort_as_half((unsigned short)0);
            const uint32_t m = ((1u << BITS) - 1u) << (BITS * (e % CW));
            if (e / CW == 0) keep0 &= ~m;
            else keep1 &= ~m;
            keepm &= ~(1u << e);
          }
      }
      if constexpr (BITS == 3) {
        // two planes: the low two bits of channels c8 .. c8 + 7 at bytes 2 cl,
        // 2 cl + 1 (a 2-bit row), their high bits in unit 2 (m mod 4) + h of
        // the high plane (m = cl / 2, h = cl mod 2, set m / 4); the lanes of
        // the two sets of a unit (cl and cl ^ 8) merge their bits
        const int m = cl >> 1, hh = cl & 1, s3 = m >> 2;
        (void)keepm;
#pragma unroll 2
        for (int k = 0; k < 16; ++k) {
          smem8<DT>(&s_in[(2 * k + par) * CPR + cl * CPE], x);
          uint32_t lo = 0u, hb = 0u;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(x[i]);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int e = 2 * i + u;
              const float xv = u ? f.y : f.x;
              uint32_t c = safe ? code_bits(xv, zf[e], sf[e], inv[e]) - kRoundMagicBits
                                : exact_code(xv, zf[e], sf[e], L);
              if constexpr (OUTL) c = ((keepm >> e) & 1u) ? c : 0u;
              lo |= (c & 3u) << (2 * e);
              hb |= (c >> 2) << hi_bit3(s3, e);
            }
          }
          hb |= __shfl_xor_sync(kFull, hb, 8);
          uint8_t* row = &s_codes[(2 * k + par) * RB];
          *reinterpret_cast<uint16_t*>(row + 2 * cl) = (uint16_t)lo;
          if (s3 == 0) *reinterpret_cast<uint16_t*>(row + kHiPlane3 + 4 * (m & 3) + 2 * hh) = (uint16_t)hb;
        }
      } else if (safe) {
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          smem8<DT>(&s_in[(2 * k + par) * CPR + cl * CPE], x);
          uint32_t acc[2] = {0u, 0u};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(x[i]);
            const int e0 = 2 * i, e1 = 2 * i + 1;
            acc[e0 / CW] += code_bits(f.x, zf[e0], sf[e0], inv[e0]) << (BITS * (e0 % CW));
            acc[e1 / CW] += code_bits(f.y, zf[e1], sf[e1], inv[e1]) << (BITS * (e1 % CW));
          }
          uint2 cw = make_uint2(acc[0] - C, acc[1] - C);
          if constexpr (OUTL) cw = make_uint2(cw.x & keep0, cw.y & keep1);
          store_key_slice<BITS>(&s_codes[(2 * k + par) * RB + cl * BITS], cw);
        }
      } else {
        // a channel group with an fp16-subnormal scale: IEEE division + clamp
        for (int k = 0; k < 16; ++k) {
          smem8<DT>(&s_in[(2 * k + par) * CPR + cl * CPE], x);
          const uint2 ex = exact_key_slice<BITS>(h2x4_bits(x), zf, sf);
          store_key_slice<BITS>(&s_codes[(2 * k + par) * RB + cl * BITS],
                                OUTL ? make_uint2(ex.x & keep0, ex.y & keep1) : ex);
        }
      }
      __syncwarp();
      uint8_t* tile = tile_at<BITS>(cv, unit, chunk);
      uint4* gdst = reinterpret_cast<uint4*>(tile + kOffKc<BITS>);
      const uint4* ssrc = reinterpret_cast<const uint4*>(s_codes);
      constexpr int CPRB = RB / 16;  // 16-byte chunks per code row
#pragma unroll
      for (int i = lane; i < 32 * CPRB; i += 32)
        gdst[(i / CPRB) * CPRB + krow_chunk<BITS>(i / CPRB, i % CPRB)] = ssrc[i];
      if constexpr (OUTL) {
        // the outlier block: channel indices, then row `lane`'s kept fp16 values
        uint8_t* ob = tile + kTileBytes<BITS>;
#pragma unroll
        for (int o = 0; o < kMaxOutliers; ++o)
          if (o < cv.n_out) {
            __half2 xr[4];
            smem8<DT>(&s_in[lane * CPR + (och[o] >> 3) * CPE], xr);
            reinterpret_cast<__half*>(ob + 16)[lane * cv.n_out + o] = pick_half(xr, och[o] & 7);
          }
        if (lane == 0) {
          uint32_t iw = 0;
#pragma unroll
          for (int o = 0; o < kMaxOutliers; ++o)
            if (o < cv.n_out) iw |= (uint32_t)och[o] << (8 * o);
          *reinterpret_cast<uint4*>(ob) = make_uint4(iw, 0u, 0u, 0u);
        }
      }
      {
        // scales (lanes of parity 0) and zeros (parity 1), in the tile's
        // channel-pair order (kscale_pos); the 16-byte store lands at c8 either way
        __half v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = par == 0 ? gp[e].sh : gp[e].zh;
        uint32_t w[4];
        if constexpr (BITS == 2 || BITS == 3) {
          // pair block m = this lane's 8 channels and its neighbour's (cl ^ 1):
          // word i = (channel 16m + i, 16m + 8 + i); the lower lane writes
          // words 0..3, the upper one words 4..7, each sending the other the
          // four values it lacks
          const int hi = cl & 1;
          const uint32_t s0 = hi ? pack_halves(v[0], v[1]) : pack_halves(v[4], v[5]);
          const uint32_t s1 = hi ? pack_halves(v[2], v[3]) : pack_halves(v[6], v[7]);
          const uint32_t r0 = __shfl_xor_sync(kFull, s0, 1), r1 = __shfl_xor_sync(kFull, s1, 1);
          const __half o[4] = {__ushort_as_half((unsigned short)(r0 & 0xffffu)),
                               __ushort_as_half((unsigned short)(r0 >> 16)),
                               __ushort_as_half((unsigned short)(r1 & 0xffffu)),
                               __ushort_as_half((unsigned short)(r1 >> 16))};
#pragma unroll
          for (int i = 0; i < 4; ++i) w[i] = hi ? pack_halves(o[i], v[4 + i]) : pack_halves(v[i], o[i]);
        } else if constexpr (BITS == 4) {
          // pair block m = this lane's 8 channels: word i = (8m + i, 8m + 4 + i)
#pragma unroll
          for (int i = 0; i < 4; ++i) w[i] = pack_halves(v[i], v[4 + i]);
        } else {
          // pair blocks 2cl, 2cl + 1 of 4 channels: word i = (4m + i, 4m + 2 + i)
          w[0] = pack_halves(v[0], v[2]);
          w[1] = pack_halves(v[1], v[3]);
          w[2] = pack_halves(v[4], v[6]);
          w[3] = pack_halves(v[5], v[7]);
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(tile + (par ? kOffZk : kOffSk<BITS>)) + c8) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      // keys of a chunk that is not a whole quantized group stay fp16
      for (int k = 0; k < 16; ++k) {
        const int t = t0 + 2 * k + par;
        if (t >= kring && t < T) {
          __half2 x[4];
          smem8<DT>(&s_in[(2 * k + par) * CPR + cl * CPE], x);
          *reinterpret_cast<uint4*>(cv.ring_k + (unit * cv.W + t % cv.W) * kHeadDim + c8) = h2x4_bits(x);
        }
      }
    }
  } else {
    // ---------------- values ----------------
    const int g = lane & 3, tl = lane >> 2;
    constexpr int CPW = 32 / BITS;  // codes per 32-bit word
    constexpr uint32_t C = magic_sum(CPW, BITS);
#pragma unroll 1
    for (int rr = 0; rr < 4; ++rr) {
      const int row = 8 * rr + tl;
      const int t = t0 + row;
      if (t >= T) continue;
      __half2 x[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) smem8<DT>(&s_in[row * CPR + vswz<CPG>(row, g * CPG + j * CPE)], x[j]);
      if (t >= vlo && t < vhi) {
        __half2 mn = x[0][0], mx = x[0][0];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mn = __hmin2(mn, x[j][i]);
            mx = __hmax2(mx, x[j][i]);
          }
        const GroupParams p = group_params(fminf(__low2float(mn), __high2float(mn)),
                                           fmaxf(__low2float(mx), __high2float(mx)), L);
        const FastParams f = fast_params(p);
        if constexpr (BITS == 3) {
          // low two bits as the 2-bit row's units of group g; high bits of
          // channels 4w + c of group g at unit w, bit hi_bit3(g / 2, 4 (g
          // mod 2) + c), merged over the row's four lanes (one per group)
          uint32_t lo[2] = {0u, 0u}, hw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 fv = __half22float2(x[e >> 3][(e & 7) >> 1]);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int ee = e + u, w = ee >> 2, c = ee & 3;
              const float xv = u ? fv.y : fv.x;
              const uint32_t q = f.safe ? code_bits(xv, p.z, p.s, f.inv) - kRoundMagicBits
                                        : exact_code(xv, p.z, p.s, L);
              lo[ee >> 4] |= (q & 3u) << (2 * (ee & 15));
              hw[w >> 1] |= (q >> 2) << (hi_bit3(g >> 1, 4 * (g & 1) + c) + 16 * (w & 1));
            }
          }
          const unsigned rmask = 0xfu << (lane & 28);  // the row's four lanes
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hw[j] |= __shfl_xor_sync(rmask, hw[j], 1);
            hw[j] |= __shfl_xor_sync(rmask, hw[j], 2);
          }
          store_value_units<2>(&s_codes[row * RB], g, lo);
          if (g == 0) *reinterpret_cast<uint4*>(&s_codes[row * RB + kHiPlane3]) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        } else {
        uint32_t words[BITS];
        if (f.safe) {
#pragma unroll
          for (int w = 0; w < BITS; ++w) {
            uint32_t acc = 0;
#pragma unroll
            for (int e2 = 0; e2 < CPW / 2; ++e2) {
              const int e = w * CPW + 2 * e2;  // channel within the group
              const float2 fv = __half22float2(x[e >> 3][(e & 7) >> 1]);
              acc += code_bits(fv.x, p.z, p.s, f.inv) << (BITS * (2 * e2));
              acc += code_bits(fv.y, p.z, p.s, f.inv) << (BITS * (2 * e2 + 1));
            }
            words[w] = acc - C;
          }
        } else {  // fp16-subnormal scale: IEEE division + clamp
          uint32_t xw[16];
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) xw[4 * j + i] = h2_bits(x[j][i]);
          exact_value_group<BITS>(xw, p.z, p.s, words);
        }
        store_value_units<BITS>(&s_codes[row * RB], g, words);
        }
        uint8_t* tile = tile_at<BITS>(cv, unit, chunk);
        reinterpret_cast<__half*>(tile + kOffSv<BITS>)[vscale_pos(row, g)] = p.sh;
        reinterpret_cast<__half*>(tile + kOffZv<BITS>)[vscale_pos(row, g)] = p.zh;
      } else if (t >= vring) {
        __half* dst = cv.ring_v + (unit * cv.W + t % cv.W) * kHeadDim + 32 * g;
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(dst + 8 * j) = h2x4_bits(x[j]);
      }
    }
    __syncwarp();
    const int r_lo = min(max(vlo - t0, 0), 32), r_hi = min(max(vhi - t0, 0), 32);
    uint4* gdst = reinterpret_cast<uint4*>(tile_at<BITS>(cv, unit, chunk) + kOffVc<BITS>);
    const uint4* ssrc = reinterpret_cast<const uint4*>(s_codes);
    constexpr int CPRB = RB / 16;  // 16-byte chunks per code row
    for (int i = r_lo * CPRB + lane; i < r_hi * CPRB; i += 32)
      gdst[(i / CPRB) * CPRB + vrow_chunk<BITS>(i / CPRB, i % CPRB)] = ssrc[i];
  }
}

// Prefill: one CTA per (32-token chunk, kv-head, b) stages the chunk's raw
// key rows (warp 0) and value rows (warp 1) with cp.async and quantizes them
// (keys of whole groups below nq_k, values below nq_v; the rest to the ring).
template <int BITS, int DT, bool OUTL>
__global__ void __launch_bounds__(64)
quantize_prefill_kernel(CacheView cv, const void* __restrict__ kin,
                        const void* __restrict__ vin, int t_in, int T_u, int nqk_u, int nqv_u,
                        const SeqLens lens) {
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int EB = DT == kF32 ? 4 : 2;
  constexpr int CPR = kHeadDim * EB / 16;
  constexpr int CPG = CPR / 4;
  __shared__ __align__(16) uint4 s_in_all[2][32 * CPR];
  __shared__ __align__(16) uint8_t s_codes_all[2][32 * RB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* s_in = s_in_all[warp];
  uint8_t* s_codes = s_codes_all[warp];
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long unit = (long)b * cv.H + h;
  const int t0 = chunk * 32;
  // this sequence's tokens: the first T of the t_in input rows.  A uniform
  // batch passes T and its counts as plain arguments (reading them from the
  // lengths parameter cost this kernel a few percent).
  int T = T_u, nq_k = nqk_u, nq_v = nqv_u;
  if (T_u < 0) {
    T = lens.l[b];
    if (t0 >= T) return;
    nq_k = policy_nq_k(T, cv.R, cv.policy);
    nq_v = policy_nq_v(T, cv.R, cv.policy);
  }
  const int rows = min(32, T - t0);
  {
    const char* src = static_cast<const char*>(warp == 0 ? kin : vin) + (unit * t_in + t0) * (long)(kHeadDim * EB);
    for (int i = lane; i < rows * CPR; i += 32) {
      const int r = i / CPR, c = i % CPR;
      cp_async16(&s_in[r * CPR + (warp == 0 ? c : vswz<CPG>(r, c))], src + 16L * i);
    }
    asm volatile("cp.async.commit_group;");
    asm volatile("cp.async.wait_group 0;");
    __syncwarp();
  }
  quantize_chunk<BITS, DT, OUTL>(cv, s_in, s_codes, unit, chunk, T, t0 + 32 <= nq_k, nq_k, 0, nq_v, nq_v);
}

// Appending n tokens to a cache of length l0 (L = l0 + n), step 1: the key
// groups that become whole, [nq_k0, nq_k1), and the value tokens that leave
// the window, [nq_v0, nq_v1), are quantized from the chunks that hold them.
// A token t < l0 is read from its ring slot, t >= l0 from the input (rounded
// to fp16).  Nothing is written to the ring (step 2 does that after every
// read of this step).  One CTA per (chunk c_lo + blockIdx.x, kv-head, b).
template <int BITS, int DT, bool OUTL>
__global__ void __launch_bounds__(64)
append_quantize_kernel(CacheView cv, const void* __restrict__ kin, const void* __restrict__ vin, int n, int c_lo,
                       const SeqLens lens) {
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int CPR = 16;  // staged as fp16: 16-byte chunks per row
  __shared__ __align__(16) uint4 s_in_all[2][32 * CPR];
  __shared__ __align__(16) uint8_t s_codes_all[2][32 * RB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* s_in = s_in_all[warp];
  uint8_t* s_codes = s_codes_all[warp];
  const int chunk = c_lo + blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long unit = (long)b * cv.H + h;
  const int t0 = chunk * 32;
  const int l0 = seq_len(lens, b), L = l0 + n;
  int cnt[4];
  seq_counts(lens, b, cv.R, cv.policy, cnt);
  const int nq_k0 = cnt[0], nq_v0 = cnt[1], nq_k1 = cnt[2], nq_v1 = cnt[3];
  // this sequence's chunks: those holding [min(nq_k0, nq_v0), max(nq_k1, nq_v1))
  const int lo = min(nq_k0, nq_v0), hi = max(nq_k1, nq_v1);
  if (hi <= lo || t0 + 32 <= lo || t0 >= hi) return;
  const int rows = min(32, L - t0);
  const __half* ring = warp == 0 ? cv.ring_k : cv.ring_v;
  const void* in = warp == 0 ? kin : vin;
  for (int i = lane; i < rows * CPR; i += 32) {
    const int r = i / CPR, c = i % CPR;
    const int t = t0 + r;
    uint4 x;
    if (t < l0) {
      x = *reinterpret_cast<const uint4*>(ring + (unit * cv.W + t % cv.W) * kHeadDim + 8 * c);
    } else {
      __half2 hx[4];
      load8<DT>(in, (unit * n + (t - l0)) * kHeadDim + 8 * c, hx);
      x = h2x4_bits(hx);
    }
    s_in[r * CPR + (warp == 0 ? c : vswz<4>(r, c))] = x;
  }
  __syncwarp();
  const bool kq = t0 >= nq_k0 && t0 + 32 <= nq_k1;
  quantize_chunk<BITS, kF16, OUTL>(cv, s_in, s_codes, unit, chunk, L, kq, INT_MAX, max(nq_v0, t0), nq_v1,
                                   INT_MAX);
}

// Appending n tokens, step 2: the last min(n, W) of them go to their ring
// slots (t mod W), keys and values, rounded to fp16.  One CTA per (token,
// kv-head, b); thread d owns channel d.
template <int DT>
__global__ void __launch_bounds__(128)
append_ring_kernel(CacheView cv, const void* __restrict__ kin, const void* __restrict__ vin, int n,
                   const SeqLens lens, int trig) {
  // a decode step's attention may start its prologue (trig); otherwise no
  // dependent launch starts before this kernel completes
  if (trig) grid_launch_dependents();
  const int m = min(n, cv.W);
  const int i = n - m + blockIdx.x;  // input row
  const int h = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const int t = seq_len(lens, b) + i;
  const long unit = (long)b * cv.H + h;
  const long src = (unit * n + i) * kHeadDim + d;
  const long dst = (unit * cv.W + t % cv.W) * kHeadDim + d;
  cv.ring_k[dst] = load1<DT>(kin, src);
  cv.ring_v[dst] = load1<DT>(vin, src);
}

// One CTA per (kv-head, b); thread d owns channel d.  Appends token t:
//  1. if t >= R, the value token t-R (in the slot t is about to take) leaves
//     the window: quantize it per token (one warp = one 32-channel group);
//  2. write k_t, v_t to ring slot t mod R;
//  3. if t+1 is a multiple of R, the key ring holds R whole groups of tokens
//     t+1-R .. t in slot order: quantize each channel of each group.
template <int BITS, int DT>
__global__ void __launch_bounds__(128)
append_kernel(CacheView cv, const void* __restrict__ kin, const void* __restrict__ vin, const SeqLens lens,
              int trig) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int PER_BYTE = 8 / BITS;
  // trig: a decode step's attention may start its prologue at once; with
  // trig 0 no dependent launch starts before this kernel completes
  if (trig) grid_launch_dependents();
  const int h = blockIdx.x, b = blockIdx.y;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const long unit = (long)b * cv.H + h;
  const int t = seq_len(lens, b);  // the new token's position in its sequence
  const int R = cv.R, slot = t % R;
  const __half kx = load1<DT>(kin, unit * kHeadDim + d);
  const __half vx = load1<DT>(vin, unit * kHeadDim + d);
  __half* ringk = cv.ring_k + unit * R * kHeadDim;
  __half* ringv = cv.ring_v + unit * R * kHeadDim;

  if (t >= R) {
    const long u = t - R;
    const float x = __half2float(ringv[slot * kHeadDim + d]);
    float mn = x, mx = x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(kFull, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    }
    const GroupParams p = group_params(mn, mx, L);
    uint8_t* tile = tile_at<BITS>(cv, unit, u / kGroup);
    const int row = (int)(u % kGroup);
    if constexpr (BITS == 3) {
      // the low two bits as a 2-bit row (unit d / 4 interleaved); the high
      // bit of channel d at unit (d mod 32) / 4, bit hi_bit3(gp / 2, 4 (gp mod
      // 2) + d mod 4) with gp = d / 32, merged over the four groups
      __shared__ uint32_t s_vh[4];
      if (d < 4) s_vh[d] = 0u;
      __syncthreads();
      const uint32_t c = encode(x, p, L);
      uint32_t q = (c & 3u) << (2 * (d & 3));
      q |= __shfl_xor_sync(kFull, q, 1);
      q |= __shfl_xor_sync(kFull, q, 2);
      if ((d & 3) == 0) tile[kOffVc<BITS> + row * RB + v_unit_pos(d / 4)] = (uint8_t)q;
      const int w = (d & 31) >> 2;
      if (c >> 2) atomicOr(&s_vh[w >> 1], 1u << (hi_bit3(warp >> 1, 4 * (warp & 1) + (d & 3)) + 16 * (w & 1)));
      __syncthreads();
      if (d < 4) reinterpret_cast<uint32_t*>(tile + kOffVc<BITS> + row * RB + kHiPlane3)[d] = s_vh[d];
    } else {
      uint32_t q = encode(x, p, L) << (BITS * (d % PER_BYTE));
#pragma unroll
      for (int off = 1; off < PER_BYTE; off <<= 1) q |= __shfl_xor_sync(kFull, q, off);
      // value rows are group-interleaved: channel d is in unit d / 4
      const int vbyte = v_unit_pos(d / 4) * (BITS / 2) + (d % 4) / PER_BYTE;
      if (d % PER_BYTE == 0) tile[kOffVc<BITS> + row * RB + vrow_byte<BITS>(row, vbyte)] = (uint8_t)q;
    }
    if (lane == 0) {
      reinterpret_cast<__half*>(tile + kOffSv<BITS>)[vscale_pos(row, warp)] = p.sh;
      reinterpret_cast<__half*>(tile + kOffZv<BITS>)[vscale_pos(row, warp)] = p.zh;
    }
  }
  // the same thread read the slot above, so program order protects it
  ringk[slot * kHeadDim + d] = kx;
  ringv[slot * kHeadDim + d] = vx;

  if ((t + 1) % R == 0) {
    const int tb = t + 1 - R;  // first ring token, in slot 0
    for (int gi = 0; gi < R / kGroup; ++gi) {
      float xs[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) xs[j] = __half2float(ringk[(gi * kGroup + j) * kHeadDim + d]);
      float mn = xs[0], mx = xs[0];
#pragma unroll
      for (int j = 1; j < kGroup; ++j) {
        mn = fminf(mn, xs[j]);
        mx = fmaxf(mx, xs[j]);
      }
      GroupParams p = group_params(mn, mx, L);
      uint8_t* tile = tile_at<BITS>(cv, unit, tb / kGroup + gi);
      // outlier-aware keys: the n_out channels with the largest max |k| of
      // the group (largest first, ties to the lower channel) stay fp16
      int slot = -1;  // this channel's place among the outliers
      if (cv.n_out > 0) {
        __shared__ float s_bv[4];
        __shared__ int s_bc[4];
        __shared__ int s_ch[kMaxOutliers];
        const float am = fmaxf(fabsf(mn), fabsf(mx));
        for (int o = 0; o < cv.n_out; ++o) {
          float bv = slot >= 0 ? -1.0f : am;
          int bc = d;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, off);
            const int oc = __shfl_xor_sync(kFull, bc, off);
            if (ov > bv || (ov == bv && oc < bc)) {
              bv = ov;
              bc = oc;
            }
          }
          if (lane == 0) {
            s_bv[warp] = bv;
            s_bc[warp] = bc;
          }
          __syncthreads();
          if (d == 0) {
            float v = s_bv[0];
            int c = s_bc[0];
            for (int w = 1; w < 4; ++w)
              if (s_bv[w] > v || (s_bv[w] == v && s_bc[w] < c)) {
                v = s_bv[w];
                c = s_bc[w];
              }
            s_ch[o] = c;
          }
          __syncthreads();
          if (s_ch[o] == d) slot = o;
        }
        if (slot >= 0) {
          p.sh = __ushort_as_half((unsigned short)0);
          p.zh = __ushort_as_half((unsigned short)0);
          __half* ov = reinterpret_cast<__half*>(tile + kTileBytes<BITS> + 16);
          for (int j = 0; j < kGroup; ++j) ov[j * cv.n_out + slot] = ringk[(gi * kGroup + j) * kHeadDim + d];
        }
        if (d == 0) {
          uint32_t iw = 0;
          for (int o = 0; o < cv.n_out; ++o) iw |= (uint32_t)s_ch[o] << (8 * o);
          *reinterpret_cast<uint4*>(tile + kTileBytes<BITS>) = make_uint4(iw, 0u, 0u, 0u);
        }
      }
      if constexpr (BITS == 3) {
        // the low two bits as a 2-bit row; the high bit of channel d = 16 m +
        // 8 h + i at unit 2 (m mod 4) + h, bit hi_bit3(m / 4, i), merged over
        // the CTA in shared memory
        __shared__ uint32_t s_kh[kGroup][4];
        for (int i = d; i < kGroup * 4; i += kHeadDim) (&s_kh[0][0])[i] = 0u;
        __syncthreads();
        const int m = d >> 4;
        const int hpos = hi_bit3(m >> 2, d & 7) + 16 * ((d >> 3) & 1);
#pragma unroll 4
        for (int j = 0; j < kGroup; ++j) {
          const uint32_t c = slot >= 0 ? 0u : encode(xs[j], p, L);
          uint32_t q = (c & 3u) << (2 * (d & 3));
          q |= __shfl_xor_sync(kFull, q, 1);
          q |= __shfl_xor_sync(kFull, q, 2);
          if ((d & 3) == 0) tile[kOffKc<BITS> + j * RB + (d >> 2)] = (uint8_t)q;
          if (c >> 2) atomicOr(&s_kh[j][m & 3], 1u << hpos);
        }
        __syncthreads();
        reinterpret_cast<uint32_t*>(tile + kOffKc<BITS> + (d >> 2) * RB + kHiPlane3)[d & 3] = s_kh[d >> 2][d & 3];
        __syncthreads();  // s_kh is cleared again by the next group
      } else {
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          uint32_t q = (slot >= 0 ? 0u : encode(xs[j], p, L)) << (BITS * (d % PER_BYTE));
#pragma unroll
          for (int off = 1; off < PER_BYTE; off <<= 1) q |= __shfl_xor_sync(kFull, q, off);
          if (d % PER_BYTE == 0) tile[kOffKc<BITS> + j * RB + krow_byte<BITS>(j, d / PER_BYTE)] = (uint8_t)q;
        }
      }
      reinterpret_cast<__half*>(tile + kOffSk<BITS>)[kscale_pos<BITS>(d)] = p.sh;
      reinterpret_cast<__half*>(tile + kOffZk)[kscale_pos<BITS>(d)] = p.zh;
      if (cv.n_out > 0) __syncthreads();  // s_ch is reused by the next group
    }
  }
}

template <int BITS>
cudaError_t prefill_bits(const CacheView& cv, const void* k, const void* v, int dtype, int t_in,
                         const SeqLens& lens, cudaStream_t st) {
  const dim3 grid((t_in + 31) / 32, cv.H, cv.B);
  const int tu = lens.uniform;
  // plain caches run the chunk quantizer without the outlier selection
  if (cv.n_out > 0) {
    switch (dtype) {
      case kF32: quantize_prefill_kernel<BITS, kF32, true><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
      case kF16: quantize_prefill_kernel<BITS, kF16, true><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
      default: quantize_prefill_kernel<BITS, kBF16, true><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
    }
  } else {
    switch (dtype) {
      case kF32: quantize_prefill_kernel<BITS, kF32, false><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
      case kF16: quantize_prefill_kernel<BITS, kF16, false><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
      default: quantize_prefill_kernel<BITS, kBF16, false><<<grid, 64, 0, st>>>(cv, k, v, t_in, tu, lens.u_nq[0], lens.u_nq[1], lens); break;
    }
  }
  return cudaGetLastError();
}

template <int BITS>
cudaError_t append_bits(const CacheView& cv, const void* k, const void* v, int dtype, const SeqLens& lens,
                        cudaStream_t st, int trig) {
  const dim3 grid(cv.H, cv.B);
  switch (dtype) {
    case kF32: append_kernel<BITS, kF32><<<grid, kHeadDim, 0, st>>>(cv, k, v, lens, trig); break;
    case kF16: append_kernel<BITS, kF16><<<grid, kHeadDim, 0, st>>>(cv, k, v, lens, trig); break;
    default: append_kernel<BITS, kBF16><<<grid, kHeadDim, 0, st>>>(cv, k, v, lens, trig); break;
  }
  return cudaGetLastError();
}

template <int BITS, int DT>
cudaError_t append_tokens_dt(const CacheView& cv, const void* k, const void* v, int n, int c_lo, int c_hi,
                             const SeqLens& lens, cudaStream_t st, int trig) {
  if (c_hi > c_lo) {
    const dim3 grid(c_hi - c_lo, cv.H, cv.B);
    if (cv.n_out > 0) append_quantize_kernel<BITS, DT, true><<<grid, 64, 0, st>>>(cv, k, v, n, c_lo, lens);
    else append_quantize_kernel<BITS, DT, false><<<grid, 64, 0, st>>>(cv, k, v, n, c_lo, lens);
  }
  append_ring_kernel<DT><<<dim3(min(n, cv.W), cv.H, cv.B), kHeadDim, 0, st>>>(cv, k, v, n, lens, trig);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t append_tokens_bits(const CacheView& cv, const void* k, const void* v, int dtype, int n, int c_lo,
                               int c_hi, const SeqLens& lens, cudaStream_t st, int trig) {
  switch (dtype) {
    case kF32: return append_tokens_dt<BITS, kF32>(cv, k, v, n, c_lo, c_hi, lens, st, trig);
    case kF16: return append_tokens_dt<BITS, kF16>(cv, k, v, n, c_lo, c_hi, lens, st, trig);
    default: return append_tokens_dt<BITS, kBF16>(cv, k, v, n, c_lo, c_hi, lens, st, trig);
  }
}

}  // namespace

cudaError_t launch_append_tokens(const CacheView& cv, const void* k, const void* v, int dtype, int n,
                                 const SeqLens& lens, cudaStream_t st, int trig) {
  if (n <= 0) return cudaSuccess;
  // the chunks holding some sequence's [min(nq_k0, nq_v0), max(nq_k1, nq_v1))
  int c_lo = INT_MAX, c_hi = 0;
  const int nb = lens.uniform >= 0 ? 1 : cv.B;
  for (int b = 0; b < nb; ++b) {
    const int l0 = seq_len(lens, b), L = l0 + n;
    const int lo = min(policy_nq_k(l0, cv.R, cv.policy), policy_nq_v(l0, cv.R, cv.policy));
    const int hi = max(policy_nq_k(L, cv.R, cv.policy), policy_nq_v(L, cv.R, cv.policy));
    if (hi > lo) {
      c_lo = min(c_lo, lo / 32);
      c_hi = max(c_hi, (hi + 31) / 32);
    }
  }
  if (c_hi == 0) c_lo = 0;
  switch (cv.bits) {
    case 2: return append_tokens_bits<2>(cv, k, v, dtype, n, c_lo, c_hi, lens, st, trig);
    case 3: return append_tokens_bits<3>(cv, k, v, dtype, n, c_lo, c_hi, lens, st, trig);
    case 4: return append_tokens_bits<4>(cv, k, v, dtype, n, c_lo, c_hi, lens, st, trig);
    default: return append_tokens_bits<8>(cv, k, v, dtype, n, c_lo, c_hi, lens, st, trig);
  }
}

cudaError_t launch_quantize_prefill(const CacheView& cv, const void* k, const void* v, int dtype, int t_in,
                                    const SeqLens& lens, cudaStream_t st) {
  if (t_in <= 0) return cudaSuccess;
  switch (cv.bits) {
    case 2: return prefill_bits<2>(cv, k, v, dtype, t_in, lens, st);
    case 3: return prefill_bits<3>(cv, k, v, dtype, t_in, lens, st);
    case 4: return prefill_bits<4>(cv, k, v, dtype, t_in, lens, st);
    default: return prefill_bits<8>(cv, k, v, dtype, t_in, lens, st);
  }
}

cudaError_t launch_append(const CacheView& cv, const void* k, const void* v, int dtype, const SeqLens& lens,
                          cudaStream_t st, int trig) {
  switch (cv.bits) {
    case 2: return append_bits<2>(cv, k, v, dtype, lens, st, trig);
    case 3: return append_bits<3>(cv, k, v, dtype, lens, st, trig);
    case 4: return append_bits<4>(cv, k, v, dtype, lens, st, trig);
    default: return append_bits<8>(cv, k, v, dtype, lens, st, trig);
  }
}

}  // namespace kivi
