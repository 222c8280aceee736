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

// Weighted combine of a token's expert outputs, then either the output or the
// post-norm + scaled residual ("Reflection 发布 Beam 501B 开源模型…", section
// 专家混合模型: expert outputs combined with the normalised router weights;
// section 残差流: normalise after the sublayer, then h_k = a*h_{k-1} + b*n):
//   o[t,:] = sum_j w[t,j] * s[r] * y[r, :], r = pair_row[t,j]   (y FP32; FP32
//            sum, slot order; s = the per-row scale of y, or 1 when y_scale
//            is NULL -- the E4M3 path's activation row scales)
//   resid:  out = bf16( a * h_prev + b * RMSNorm(o) * gain )
//   else:   out = o  (bf16, or fp32 when OUT_F32)
// One block of 128 threads per token; each thread keeps up to 8 chunks of 8
// elements of o in registers (H <= 8192).
constexpr int COMBINE_THREADS = 128;
constexpr int COMBINE_MAX_CHUNKS = 8;

template <bool OUT_F32>
__global__ void __launch_bounds__(COMBINE_THREADS) combine_rows_kernel(
    const float* __restrict__ y, const float* __restrict__ y_scale, const int* __restrict__ pair_row,
    const float* __restrict__ topk_w, int top_k, const __nv_bfloat16* __restrict__ h_prev,
    const float* __restrict__ gain, void* __restrict__ out, int H, float eps, float a, float b,
    int resid) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  __shared__ float s_red[COMBINE_THREADS / 32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < top_k) {
    const int r = pair_row[static_cast<size_t>(t) * top_k + tid];
    s_row[tid] = r;
    const float wt = topk_w[static_cast<size_t>(t) * top_k + tid];
    s_w[tid] = y_scale != nullptr ? wt * y_scale[r] : wt;
  }
  __syncthreads();
  const int nc = H >> 3;
  float o[COMBINE_MAX_CHUNKS][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i) {
    const int c = tid + i * COMBINE_THREADS;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[i][e] = 0.f;
    if (c < nc) {
      for (int j = 0; j < top_k; ++j) {
        float f[8];
        load8(y + static_cast<size_t>(s_row[j]) * H, c, f);
        const float wj = s_w[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[i][e] = fmaf(wj, f[e], o[i][e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(o[i][e], o[i][e], ss);
    }
  }
  float r = 1.f;
  if (resid) {
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) tot += s_red[w];
    r = rsqrtf(tot / static_cast<float>(H) + eps);
  }
#pragma unroll
  for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i) {
    const int c = tid + i * COMBINE_THREADS;
    if (c >= nc) continue;
    if (OUT_F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<size_t>(t) * H) + 2 * c;
      dst[0] = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
      dst[1] = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
    } else {
      float f[8];
      if (resid) {
        float hv[8], g[8];
        load8(h_prev + static_cast<size_t>(t) * H, c, hv);
        gain8(gain, c, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = fmaf(a, hv[e], b * (o[i][e] * r * g[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = o[i][e];
      }
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + static_cast<size_t>(t) * H)[c] =
          f32x8_to_bf16(f);
    }
  }
}

}  // namespace beam
