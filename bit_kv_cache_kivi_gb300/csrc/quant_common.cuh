// quant_common.cuh -- the per-group min/max quantizer on the device (internal).
//
// The quantizer of the pages (veloxquant-mlx "KIVI", How it works; chooblog
// KIVI review §1.1; notebook "KIVI - 2-bit KV cache quantisation"):
//   zero = min(group), scale = (max - min) / (2^b - 1),
//   q = round((x - zero) / scale) clamped to [0, 2^b - 1].
// The scale and zero are stored as fp16 and the codes are computed with the
// stored fp16 scale; a zero range (or a scale that rounds to fp16 zero)
// stores scale 1.  Rounding is to nearest, ties to even, and every
// floating-point decision is taken in fp32 with IEEE rounding, so the codes
// are bit-identical to a plain sequential fp32 evaluation of the formula.
#pragma once

#include "kivi_internal.cuh"

namespace kivi {

// Adding 1.5 * 2^23 to 0 <= y < 2^22 leaves rint(y) (ties to even) in the low
// mantissa bits of the sum; subtracting it again gives rint(y) as a float.
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kRoundMagicBits = 0x4B400000u;
// |y - rint(y)| beyond this means y lies within 2^-12 of a rounding boundary.
constexpr float kNearHalf = 0.499755859375f;

struct GroupParams {
  float z, s, inv;
  __half zh, sh;
};

__device__ __forceinline__ GroupParams group_params(float mn, float mx, int L) {
  GroupParams p;
  const float r = __fsub_rn(mx, mn);
  const float s32 = __fdiv_rn(r, (float)L);
  p.sh = __float2half_rn(s32);
  p.s = __half2float(p.sh);
  if (r == 0.0f || p.s == 0.0f) {
    p.sh = __float2half_rn(1.0f);
    p.s = 1.0f;
  }
  // -0 and +0 compare equal; the stored zero point is canonically +0.
  p.zh = __float2half_rn(__fadd_rn(mn, 0.0f));
  p.z = __half2float(p.zh);
  p.inv = __frcp_rn(p.s);
  return p;
}

// Code of one fp16 value x (widened).  y = (x - z) * (1/s) differs from the
// IEEE quotient (x - z) / s by less than 2^-18 for y < 16, so unless y is
// within 2^-12 of a half-integer both round to the same integer; those rare
// near-ties are recomputed with the exact division.
__device__ __forceinline__ uint32_t encode(float x, const GroupParams& p, int L) {
  const float d = __fsub_rn(x, p.z);
  const float y = __fmul_rn(d, p.inv);
  const float t = __fadd_rn(y, kRoundMagic);
  const float r = __fsub_rn(t, kRoundMagic);
  int q = (int)(__float_as_uint(t) - kRoundMagicBits);
  if (fabsf(__fsub_rn(y, r)) > kNearHalf) q = __float2int_rn(__fdiv_rn(d, p.s));
  return (uint32_t)min(max(q, 0), L);
}

// ---- ingestion: input elements rounded to fp16 (nearest even) -------------

template <int DT>
__device__ __forceinline__ void load8(const void* base, long idx, __half2 (&h)[4]);

template <>
__device__ __forceinline__ void load8<kF16>(const void* base, long idx, __half2 (&h)[4]) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __half*>(base) + idx));
  h[0] = *reinterpret_cast<const __half2*>(&u.x);
  h[1] = *reinterpret_cast<const __half2*>(&u.y);
  h[2] = *reinterpret_cast<const __half2*>(&u.z);
  h[3] = *reinterpret_cast<const __half2*>(&u.w);
}

__device__ __forceinline__ __half2 bf16x2_to_half2(uint32_t w) {
  // bf16 is the upper half of an fp32 pattern: widening is exact.
  return __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <>
__device__ __forceinline__ void load8<kBF16>(const void* base, long idx, __half2 (&h)[4]) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
  h[0] = bf16x2_to_half2(u.x);
  h[1] = bf16x2_to_half2(u.y);
  h[2] = bf16x2_to_half2(u.z);
  h[3] = bf16x2_to_half2(u.w);
}

template <>
__device__ __forceinline__ void load8<kF32>(const void* base, long idx, __half2 (&h)[4]) {
  const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
  const float4 a = __ldcs(p), b = __ldcs(p + 1);
  h[0] = __floats2half2_rn(a.x, a.y);
  h[1] = __floats2half2_rn(a.z, a.w);
  h[2] = __floats2half2_rn(b.x, b.y);
  h[3] = __floats2half2_rn(b.z, b.w);
}

template <int DT>
__device__ __forceinline__ __half load1(const void* base, long idx) {
  if constexpr (DT == kF16) return static_cast<const __half*>(base)[idx];
  if constexpr (DT == kBF16)
    return __float2half_rn(__uint_as_float((uint32_t)static_cast<const uint16_t*>(base)[idx] << 16));
  return __float2half_rn(static_cast<const float*>(base)[idx]);
}

}  // namespace kivi
