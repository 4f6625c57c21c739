// quantize.cu -- prefill quantize/pack and decode append/flush kernels.
//
// Grouping (veloxquant-mlx "KIVI", How it works items 1-2; notebook "KIVI -
// 2-bit KV cache quantisation", K along dim 0 and V along dim 1 with group
// 32): keys per channel over groups of G = 32 tokens, values per token over
// groups of G = 32 channels.  Residual split (chooblog KIVI review, §3.2.2
// and Algorithm 1): the first nq_k = R*floor(l/R) keys and nq_v = max(l-R, 0)
// values are quantized, the rest stay fp16 in a ring of R slots.
#include "quant_common.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Value rows are group-interleaved: the unit of 4 channels 32*gp + 4*w .. +3
// (bits/2 bytes) is stored at unit position 4*w + gp.
__device__ __forceinline__ int v_unit_pos(int unit) { return 4 * (unit & 7) + (unit >> 3); }

__device__ __forceinline__ uint32_t pack_halves(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) {
  return pack_halves(__low2half(v), __high2half(v));
}

__device__ __forceinline__ uint4 h2x4_bits(const __half2 (&v)[4]) {
  return make_uint4(h2_bits(v[0]), h2_bits(v[1]), h2_bits(v[2]), h2_bits(v[3]));
}

// One CTA = one 32-token chunk of one (b, kv-head): warp 0 quantizes the
// chunk's keys (one K group: 128 channels x 32 tokens), warp 1 its values
// (32 tokens x 4 channel groups).  Lane l holds channels 8*(l%16) .. +7 of
// the tokens of parity l/16 (16-byte loads, a token row per half-warp).
template <int BITS, int DT>
__global__ void __launch_bounds__(64)
quantize_prefill_kernel(CacheView cv, const void* __restrict__ kin,
                        const void* __restrict__ vin, int T, int nq_k, int nq_v) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;  // packed bytes per token row
  constexpr int LB = BITS;                 // packed bytes of a lane's 8 channels
  __shared__ __align__(16) uint8_t s_codes[2][32 * RB];
  __shared__ __align__(16) __half s_sz[32][8];  // V rows: scale[4], zero[4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long unit = (long)b * cv.H + h;
  const int t0 = chunk * 32;
  const int cl = lane & 15, par = lane >> 4;
  const int c8 = cl * 8;
  const void* src = warp == 0 ? kin : vin;

  __half2 x[16][4];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int t = t0 + 2 * k + par;
    if (t < T) {
      load8<DT>(src, (unit * T + t) * kHeadDim + c8, x[k]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) x[k][i] = __float2half2_rn(0.0f);
    }
  }

  if (warp == 0) {
    if (t0 + 32 <= nq_k) {
      // ---- per-channel key group: min/max over 32 tokens ----
      __half2 mn[4], mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mn[i] = mx[i] = x[0][i];
#pragma unroll
      for (int k = 1; k < 16; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mn[i] = __hmin2(mn[i], x[k][i]);
          mx[i] = __hmax2(mx[i], x[k][i]);
        }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // the other token parity
        mn[i] = __hmin2(mn[i], __shfl_xor_sync(kFull, mn[i], 16));
        mx[i] = __hmax2(mx[i], __shfl_xor_sync(kFull, mx[i], 16));
      }
      GroupParams p[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        p[2 * i] = group_params(__low2float(mn[i]), __low2float(mx[i]), L);
        p[2 * i + 1] = group_params(__high2float(mn[i]), __high2float(mx[i]), L);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(x[k][i]);
          packed |= encode(f.x, p[2 * i], L) << (BITS * (2 * i));
          packed |= encode(f.y, p[2 * i + 1], L) << (BITS * (2 * i + 1));
        }
        uint8_t* dst = &s_codes[0][(2 * k + par) * RB + cl * LB];
        if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
        else *reinterpret_cast<uint32_t*>(dst) = packed;
      }
      __syncwarp();
      uint4* gdst = reinterpret_cast<uint4*>(cv.codes_k + (unit * cv.Tcap + t0) * RB);
      const uint4* ssrc = reinterpret_cast<const uint4*>(s_codes[0]);
#pragma unroll
      for (int i = lane; i < 32 * RB / 16; i += 32) gdst[i] = ssrc[i];
      if (par == 0) {
        const long so = (unit * (cv.Tcap / kGroup) + chunk) * kHeadDim + c8;
        *reinterpret_cast<uint4*>(cv.scale_k + so) =
            make_uint4(pack_halves(p[0].sh, p[1].sh), pack_halves(p[2].sh, p[3].sh),
                       pack_halves(p[4].sh, p[5].sh), pack_halves(p[6].sh, p[7].sh));
        *reinterpret_cast<uint4*>(cv.zero_k + so) =
            make_uint4(pack_halves(p[0].zh, p[1].zh), pack_halves(p[2].zh, p[3].zh),
                       pack_halves(p[4].zh, p[5].zh), pack_halves(p[6].zh, p[7].zh));
      }
    } else {
      // keys of a chunk that is not a whole quantized group stay fp16
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int t = t0 + 2 * k + par;
        if (t >= nq_k && t < T)
          *reinterpret_cast<uint4*>(cv.ring_k + (unit * cv.R + t % cv.R) * kHeadDim + c8) =
              h2x4_bits(x[k]);
      }
    }
  } else {
    // ---- per-token value groups: 4 lanes x 8 channels = 32 channels ----
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int t = t0 + 2 * k + par;
      const __half2 a = __hmin2(__hmin2(x[k][0], x[k][1]), __hmin2(x[k][2], x[k][3]));
      const __half2 c = __hmax2(__hmax2(x[k][0], x[k][1]), __hmax2(x[k][2], x[k][3]));
      __half2 mm = __halves2half2(__hmin(__low2half(a), __high2half(a)),
                                  __hmax(__low2half(c), __high2half(c)));
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        const __half2 o = __shfl_xor_sync(kFull, mm, off);
        mm = __halves2half2(__hmin(__low2half(mm), __low2half(o)),
                            __hmax(__high2half(mm), __high2half(o)));
      }
      if (t < nq_v) {
        const GroupParams p = group_params(__low2float(mm), __high2float(mm), L);
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(x[k][i]);
          packed |= encode(f.x, p, L) << (BITS * (2 * i));
          packed |= encode(f.y, p, L) << (BITS * (2 * i + 1));
        }
        // this lane's 8 channels are the units 2*cl and 2*cl + 1
        uint8_t* row = &s_codes[1][(2 * k + par) * RB];
        if constexpr (BITS == 2) {
          row[v_unit_pos(2 * cl)] = (uint8_t)packed;
          row[v_unit_pos(2 * cl + 1)] = (uint8_t)(packed >> 8);
        } else {
          reinterpret_cast<uint16_t*>(row)[v_unit_pos(2 * cl)] = (uint16_t)packed;
          reinterpret_cast<uint16_t*>(row)[v_unit_pos(2 * cl + 1)] = (uint16_t)(packed >> 16);
        }
        if ((lane & 3) == 0) {
          s_sz[2 * k + par][cl >> 2] = p.sh;
          s_sz[2 * k + par][4 + (cl >> 2)] = p.zh;
        }
      } else if (t < T) {
        *reinterpret_cast<uint4*>(cv.ring_v + (unit * cv.R + t % cv.R) * kHeadDim + c8) =
            h2x4_bits(x[k]);
      }
    }
    __syncwarp();
    const int nrows = min(max(nq_v - t0, 0), 32);
    if (nrows > 0) {
      uint4* gdst = reinterpret_cast<uint4*>(cv.codes_v + (unit * cv.Tcap + t0) * RB);
      const uint4* ssrc = reinterpret_cast<const uint4*>(s_codes[1]);
      for (int i = lane; i < nrows * RB / 16; i += 32) gdst[i] = ssrc[i];
      if (lane < nrows) {
        const long so = (unit * cv.Tcap + t0 + lane) * (kHeadDim / kGroup);
        *reinterpret_cast<uint2*>(cv.scale_v + so) = *reinterpret_cast<const uint2*>(&s_sz[lane][0]);
        *reinterpret_cast<uint2*>(cv.zero_v + so) = *reinterpret_cast<const uint2*>(&s_sz[lane][4]);
      }
    }
  }
}

// One CTA per (kv-head, b); thread d owns channel d.  Appends token t:
//  1. if t >= R, the value token t-R (in the slot t is about to take) leaves
//     the window: quantize it per token (one warp = one 32-channel group);
//  2. write k_t, v_t to ring slot t mod R;
//  3. if t+1 is a multiple of R, the key ring holds R whole groups of tokens
//     t+1-R .. t in slot order: quantize each channel of each group.
template <int BITS, int DT>
__global__ void __launch_bounds__(128)
append_kernel(CacheView cv, const void* __restrict__ kin, const void* __restrict__ vin, int t) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int PER_BYTE = 8 / BITS;
  const int h = blockIdx.x, b = blockIdx.y;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const long unit = (long)b * cv.H + h;
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
    uint32_t q = encode(x, p, L) << (BITS * (d % PER_BYTE));
#pragma unroll
    for (int off = 1; off < PER_BYTE; off <<= 1) q |= __shfl_xor_sync(kFull, q, off);
    // value rows are group-interleaved: channel d is in unit d / 4
    const int vbyte = v_unit_pos(d / 4) * (BITS / 2) + (d % 4) / PER_BYTE;
    if (d % PER_BYTE == 0) cv.codes_v[(unit * cv.Tcap + u) * RB + vbyte] = (uint8_t)q;
    if (lane == 0) {
      cv.scale_v[(unit * cv.Tcap + u) * (kHeadDim / kGroup) + warp] = p.sh;
      cv.zero_v[(unit * cv.Tcap + u) * (kHeadDim / kGroup) + warp] = p.zh;
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
      const GroupParams p = group_params(mn, mx, L);
      const long row0 = unit * cv.Tcap + tb + gi * kGroup;
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        uint32_t q = encode(xs[j], p, L) << (BITS * (d % PER_BYTE));
#pragma unroll
        for (int off = 1; off < PER_BYTE; off <<= 1) q |= __shfl_xor_sync(kFull, q, off);
        if (d % PER_BYTE == 0) cv.codes_k[(row0 + j) * RB + d / PER_BYTE] = (uint8_t)q;
      }
      const long so = (unit * (cv.Tcap / kGroup) + tb / kGroup + gi) * kHeadDim + d;
      cv.scale_k[so] = p.sh;
      cv.zero_k[so] = p.zh;
    }
  }
}

template <int BITS>
cudaError_t prefill_bits(const CacheView& cv, const void* k, const void* v, int dtype,
                         int T, int nq_k, int nq_v, cudaStream_t st) {
  const dim3 grid((T + 31) / 32, cv.H, cv.B);
  switch (dtype) {
    case kF32: quantize_prefill_kernel<BITS, kF32><<<grid, 64, 0, st>>>(cv, k, v, T, nq_k, nq_v); break;
    case kF16: quantize_prefill_kernel<BITS, kF16><<<grid, 64, 0, st>>>(cv, k, v, T, nq_k, nq_v); break;
    default: quantize_prefill_kernel<BITS, kBF16><<<grid, 64, 0, st>>>(cv, k, v, T, nq_k, nq_v); break;
  }
  return cudaGetLastError();
}

template <int BITS>
cudaError_t append_bits(const CacheView& cv, const void* k, const void* v, int dtype, int t,
                        cudaStream_t st) {
  const dim3 grid(cv.H, cv.B);
  switch (dtype) {
    case kF32: append_kernel<BITS, kF32><<<grid, kHeadDim, 0, st>>>(cv, k, v, t); break;
    case kF16: append_kernel<BITS, kF16><<<grid, kHeadDim, 0, st>>>(cv, k, v, t); break;
    default: append_kernel<BITS, kBF16><<<grid, kHeadDim, 0, st>>>(cv, k, v, t); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_prefill(const CacheView& cv, const void* k, const void* v,
                                    int dtype, int T, int nq_k, int nq_v, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  return cv.bits == 2 ? prefill_bits<2>(cv, k, v, dtype, T, nq_k, nq_v, st)
                      : prefill_bits<4>(cv, k, v, dtype, T, nq_k, nq_v, st);
}

cudaError_t launch_append(const CacheView& cv, const void* k, const void* v, int dtype, int t,
                          cudaStream_t st) {
  return cv.bits == 2 ? append_bits<2>(cv, k, v, dtype, t, st)
                      : append_bits<4>(cv, k, v, dtype, t, st);
}

}  // namespace kivi
