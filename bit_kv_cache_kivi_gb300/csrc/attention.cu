// attention.cu -- decode attention over the packed KIVI cache, split along the
// context (flash-decoding style) with the split combine fused into the same
// launch.
//
// Decode step 2 of the chooblog KIVI review (§1.3): A = softmax(t_Q X_K^T),
// t_O = A X_V, with the 1/sqrt(D) scale of the notebook "KIVI - 2-bit KV cache
// quantisation"; dequantization is fused into both products (review §3.2
// "System-Level": no separate dequantize pass).
//
// Algebra used for the packed keys of group g (32 tokens, per-channel scale
// s_d and zero z_d): q . khat_t = sum_d (q_d s_d) c_td + sum_d q_d z_d, so each
// group costs one q' = q * s and one beta = q . z per head, and a token costs
// one dot product with its small-integer codes.
#include <cuda_bf16.h>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 4;

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

__device__ __forceinline__ void halves4(uint2 u, float (&f)[4]) {
  f[0] = h_lo(u.x);
  f[1] = h_hi(u.x);
  f[2] = h_lo(u.y);
  f[3] = h_hi(u.y);
}

// grid (splits, H * head_chunks, B), 128 threads.  A CTA handles up to NH
// query heads of one KV head over the tokens of one split; each warp walks
// 32-token tiles (one key group each) with its own online softmax, and the
// four warps are merged at the end into one (max, sum, output) partial.
template <int BITS, int NH>
__global__ void __launch_bounds__(128)
attn_split_kernel(CacheView cv, AttnArgs a) {
  constexpr int L = (1 << BITS) - 1;
  constexpr int RB = kHeadDim * BITS / 8;
  constexpr int CPW = 32 / BITS;  // codes per 32-bit word
  __shared__ __align__(16) float s_q[NH][kHeadDim];
  __shared__ __align__(16) float s_qk[kWarps][NH][kHeadDim];
  __shared__ __align__(16) uint8_t s_vc[kWarps][32 * RB];
  __shared__ __align__(16) __half s_vsz[kWarps][32][8];
  __shared__ float s_m[kWarps][NH], s_l[kWarps][NH];

  const int s = blockIdx.x;
  const int nhc = gridDim.y / cv.H;
  const int h = blockIdx.y / nhc, hc = blockIdx.y % nhc;
  const int b = blockIdx.z;
  const int grp = a.Hq / cv.H;
  const int j0 = h * grp + hc * NH;
  const int nh = min(NH, grp - hc * NH);
  const long unit = (long)b * cv.H + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_begin = s * a.chunk;
  const int t_end = min(a.l, t_begin + a.chunk);

  for (int i = threadIdx.x; i < NH * kHeadDim; i += blockDim.x) {
    const int j = i / kHeadDim, d = i % kHeadDim;
    s_q[j][d] = j < nh ? load_q(a.q, ((long)b * a.Hq + j0 + j) * kHeadDim + d, a.q_dtype) * a.scale_log2
                       : 0.0f;
  }
  __syncthreads();

  float m[NH], lsum[NH], o[NH][4];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    m[j] = -INFINITY;
    lsum[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[j][i] = 0.0f;
  }

  const int tile_end = (t_end + 31) / 32;
  for (int tile = t_begin / 32 + warp; tile < tile_end; tile += kWarps) {
    const int tt0 = tile * 32;
    const int t = tt0 + lane;
    const bool valid = t < t_end;
    float sc[NH];
    if (tt0 + 32 <= a.nq_k) {
      // ---- packed keys: q' = q * sK[g] (to smem), beta = q . zK[g] ----
      const long go = (unit * (cv.Tcap / kGroup) + tile) * kHeadDim + 4 * lane;
      float skf[4], zkf[4];
      halves4(*reinterpret_cast<const uint2*>(cv.scale_k + go), skf);
      halves4(*reinterpret_cast<const uint2*>(cv.zero_k + go), zkf);
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float4 qv = *reinterpret_cast<const float4*>(&s_q[j][4 * lane]);
        *reinterpret_cast<float4*>(&s_qk[warp][j][4 * lane]) =
            make_float4(qv.x * skf[0], qv.y * skf[1], qv.z * skf[2], qv.w * skf[3]);
        sc[j] = warp_sum(qv.x * zkf[0] + qv.y * zkf[1] + qv.z * zkf[2] + qv.w * zkf[3]);
      }
      __syncwarp();
      if (valid) {
        const uint4* row = reinterpret_cast<const uint4*>(cv.codes_k + (unit * cv.Tcap + t) * RB);
#pragma unroll
        for (int w4 = 0; w4 < RB / 16; ++w4) {
          const uint4 cw = row[w4];
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const int dbase = (w4 * 4 + wi) * CPW;
#pragma unroll
            for (int e = 0; e < CPW; e += 4) {
              const float c0 = (float)((words[wi] >> (BITS * (e + 0))) & L);
              const float c1 = (float)((words[wi] >> (BITS * (e + 1))) & L);
              const float c2 = (float)((words[wi] >> (BITS * (e + 2))) & L);
              const float c3 = (float)((words[wi] >> (BITS * (e + 3))) & L);
#pragma unroll
              for (int j = 0; j < NH; ++j) {
                const float4 qk = *reinterpret_cast<const float4*>(&s_qk[warp][j][dbase + e]);
                sc[j] += qk.x * c0 + qk.y * c1 + qk.z * c2 + qk.w * c3;
              }
            }
          }
        }
      }
    } else {
      // ---- residual keys: fp16 ring ----
#pragma unroll
      for (int j = 0; j < NH; ++j) sc[j] = 0.0f;
      if (valid) {
        const __half* kr = cv.ring_k + (unit * cv.R + t % cv.R) * kHeadDim;
#pragma unroll 4
        for (int d8 = 0; d8 < kHeadDim; d8 += 8) {
          const uint4 kv = *reinterpret_cast<const uint4*>(kr + d8);
          const float kf[8] = {h_lo(kv.x), h_hi(kv.x), h_lo(kv.y), h_hi(kv.y),
                               h_lo(kv.z), h_hi(kv.z), h_lo(kv.w), h_hi(kv.w)};
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const float4 q0 = *reinterpret_cast<const float4*>(&s_q[j][d8]);
            const float4 q1 = *reinterpret_cast<const float4*>(&s_q[j][d8 + 4]);
            sc[j] += q0.x * kf[0] + q0.y * kf[1] + q0.z * kf[2] + q0.w * kf[3] +
                     q1.x * kf[4] + q1.y * kf[5] + q1.z * kf[6] + q1.w * kf[7];
          }
        }
      }
    }

    // ---- online softmax (log2 domain: q already carries scale * log2 e) ----
    float p[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      const float sj = valid ? sc[j] : -INFINITY;
      const float mnew = fmaxf(m[j], warp_max(sj));
      const float corr = fast_exp2(m[j] - mnew);
      p[j] = fast_exp2(sj - mnew);
      lsum[j] = lsum[j] * corr + p[j];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] *= corr;
      m[j] = mnew;
    }

    // ---- values: stage the packed rows of this tile, then accumulate ----
    const int vrows = min(max(a.nq_v - tt0, 0), 32);
    {
      const uint4* gsrc = reinterpret_cast<const uint4*>(cv.codes_v + (unit * cv.Tcap + tt0) * RB);
      uint4* sdst = reinterpret_cast<uint4*>(s_vc[warp]);
      for (int i = lane; i < vrows * RB / 16; i += 32) sdst[i] = gsrc[i];
      if (lane < vrows) {
        const long so = (unit * cv.Tcap + tt0 + lane) * (kHeadDim / kGroup);
        *reinterpret_cast<uint2*>(&s_vsz[warp][lane][0]) = *reinterpret_cast<const uint2*>(cv.scale_v + so);
        *reinterpret_cast<uint2*>(&s_vsz[warp][lane][4]) = *reinterpret_cast<const uint2*>(cv.zero_v + so);
      }
    }
    __syncwarp();
    const int ntok = min(32, t_end - tt0);
    for (int r = 0; r < ntok; ++r) {
      float vh[4];
      if (r < vrows) {
        uint32_t cb;
        if constexpr (BITS == 2) cb = s_vc[warp][r * RB + lane];
        else cb = *reinterpret_cast<const uint16_t*>(&s_vc[warp][r * RB + 2 * lane]);
        const float sv = __half2float(s_vsz[warp][r][lane >> 3]);
        const float zv = __half2float(s_vsz[warp][r][4 + (lane >> 3)]);
#pragma unroll
        for (int i = 0; i < 4; ++i) vh[i] = (float)((cb >> (BITS * i)) & L) * sv + zv;
      } else {
        const __half* vr = cv.ring_v + (unit * cv.R + (tt0 + r) % cv.R) * kHeadDim + 4 * lane;
        halves4(*reinterpret_cast<const uint2*>(vr), vh);
      }
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float pr = __shfl_sync(kFull, p[j], r);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[j][i] += pr * vh[i];
      }
    }
    __syncwarp();
  }

  // ---- merge the four warps ----
#pragma unroll
  for (int j = 0; j < NH; ++j) lsum[j] = warp_sum(lsum[j]);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      s_m[warp][j] = m[j];
      s_l[warp][j] = lsum[j];
    }
  }
#pragma unroll
  for (int j = 0; j < NH; ++j)
    *reinterpret_cast<float4*>(&s_qk[warp][j][4 * lane]) = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
  __syncthreads();
  const int d = threadIdx.x;
  for (int j = 0; j < nh; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][j]);
    float lt = 0.0f, ot = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = fast_exp2(s_m[w][j] - M);
        lt += e * s_l[w][j];
        ot += e * s_qk[w][j][d];
      }
    }
    const long pidx = ((long)b * a.Hq + j0 + j) * a.splits + s;
    a.ws_o[pidx * kHeadDim + d] = ot;
    if (d == 0) {
      a.ws_ml[pidx * 2] = M;
      a.ws_ml[pidx * 2 + 1] = lt;
    }
  }

  // ---- the last CTA of this (b, kv-head, head chunk) to finish merges the
  // split partials into the output.  Nothing waits: each CTA publishes its
  // partial, counts itself in, and only the one that counts last reads them.
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* counter = a.counters + (long)b * gridDim.y + blockIdx.y;
    s_last = atomicAdd(counter, 1) == a.splits - 1;
    if (s_last) *counter = 0;  // every other CTA of the group has counted in
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int j = 0; j < nh; ++j) {
    const long base = ((long)b * a.Hq + j0 + j) * a.splits;
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, __ldcg(a.ws_ml + (base + sp) * 2));
    float den = 0.0f, num = 0.0f;
    for (int sp = 0; sp < a.splits; ++sp) {
      const float ms = __ldcg(a.ws_ml + (base + sp) * 2);
      if (ms == -INFINITY) continue;
      const float e = fast_exp2(ms - M);
      den += e * __ldcg(a.ws_ml + (base + sp) * 2 + 1);
      num += e * __ldcg(a.ws_o + (base + sp) * kHeadDim + d);
    }
    const float r = num / den;
    const long oi = ((long)b * a.Hq + j0 + j) * kHeadDim + d;
    if (a.q_dtype == kF32) static_cast<float*>(a.out)[oi] = r;
    else if (a.q_dtype == kF16) static_cast<__half*>(a.out)[oi] = __float2half_rn(r);
    else static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(r);
  }
}

template <int BITS, int NH>
void launch_split(const CacheView& cv, const AttnArgs& a, int nhc, cudaStream_t st) {
  const dim3 grid(a.splits, cv.H * nhc, cv.B);
  attn_split_kernel<BITS, NH><<<grid, 128, 0, st>>>(cv, a);
}

template <int BITS>
void launch_split_bits(const CacheView& cv, const AttnArgs& a, cudaStream_t st) {
  const int grp = a.Hq / cv.H;
  if (grp <= 1) launch_split<BITS, 1>(cv, a, 1, st);
  else if (grp <= 2) launch_split<BITS, 2>(cv, a, 1, st);
  else if (grp <= 4) launch_split<BITS, 4>(cv, a, 1, st);
  else launch_split<BITS, 8>(cv, a, (grp + 7) / 8, st);
}

}  // namespace

cudaError_t launch_attention(const CacheView& cv, const AttnArgs& a, cudaStream_t st) {
  if (cv.bits == 2) launch_split_bits<2>(cv, a, st);
  else launch_split_bits<4>(cv, a, st);
  return cudaGetLastError();
}

}  // namespace kivi
