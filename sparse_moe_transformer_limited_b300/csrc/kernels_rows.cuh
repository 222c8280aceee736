// Row-wise kernels: pre-sublayer RMSNorm, and the post-sublayer RMSNorm with
// the scaled residual update ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens
// 上下文", section 残差流: every sublayer is normalised before and after; at
// step k the stream keeps weight sqrt((k-1)/k) and the sublayer output gets
// 1/sqrt(k); normalisation runs in FP32).
//
// One warp per row; 16-byte vector loads and stores. These kernels are bound
// by HBM bandwidth (a few bytes per element).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace beam {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// Eight consecutive elements of a row, from bf16 or fp32 storage.
__device__ __forceinline__ void load8(const __nv_bfloat16* row, int c, float (&f)[8]) {
  bf16x8_to_f32(reinterpret_cast<const uint4*>(row)[c], f);
}
__device__ __forceinline__ void load8(const float* row, int c, float (&f)[8]) {
  const float4* p = reinterpret_cast<const float4*>(row) + 2 * c;
  float4 a = p[0], b = p[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void gain8(const float* gain, int c, float (&g)[8]) {
  if (gain == nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 1.f;
  } else {
    const float4* p = reinterpret_cast<const float4*>(gain) + 2 * c;
    float4 a = p[0], b = p[1];
    g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
  }
}

// x[t,:] = bf16( h[t,:] / sqrt(mean(h[t,:]^2) + eps) * gain )
__global__ void __launch_bounds__(256) prenorm_kernel(const __nv_bfloat16* __restrict__ h,
                                                      const float* __restrict__ gain,
                                                      __nv_bfloat16* __restrict__ x, int T,
                                                      int H, float eps) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const __nv_bfloat16* src = h + static_cast<size_t>(row) * H;
  const int nc = H >> 3;
  float ss = 0.f;
  for (int c = lane; c < nc; c += 32) {
    float f[8];
    load8(src, c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  uint4* dst = reinterpret_cast<uint4*>(x + static_cast<size_t>(row) * H);
  for (int c = lane; c < nc; c += 32) {
    float f[8], g[8];
    load8(src, c, f);
    gain8(gain, c, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * r * g[i];
    dst[c] = f32x8_to_bf16(f);
  }
}

// Finalise rows of an FP32/BF16 sublayer output `o`:
//   resid:  out = bf16( a * h_prev + b * (norm ? RMSNorm(o) * gain : o) )
//   else:   out = bf16(o)
// `out` may alias `h_prev` (each element is read before the same thread
// writes it).
template <typename TIn>
__global__ void __launch_bounds__(256) finalize_rows_kernel(
    const TIn* __restrict__ o, const __nv_bfloat16* h_prev, const float* __restrict__ gain,
    __nv_bfloat16* out, int T, int H, float eps, float a, float b, int resid, int norm) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const TIn* src = o + static_cast<size_t>(row) * H;
  const int nc = H >> 3;
  float r = 1.f;
  if (resid && norm) {
    float ss = 0.f;
    for (int c = lane; c < nc; c += 32) {
      float f[8];
      load8(src, c, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum(ss);
    r = rsqrtf(ss / static_cast<float>(H) + eps);
  }
  const __nv_bfloat16* hp = h_prev + static_cast<size_t>(row) * H;
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * H);
  for (int c = lane; c < nc; c += 32) {
    float f[8];
    load8(src, c, f);
    if (resid) {
      float hv[8], g[8];
      load8(hp, c, hv);
      if (norm) {
        gain8(gain, c, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = f[i] * r * g[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = fmaf(a, hv[i], b * f[i]);
    }
    dst[c] = f32x8_to_bf16(f);
  }
}

}  // namespace beam
