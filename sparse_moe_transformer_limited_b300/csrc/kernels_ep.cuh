// Expert-parallel helpers: the sublayer split across P devices by expert
// ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文", section 多 GPU 和多节点:
// each expert lives on one device, the device count divides the 256 experts).
// A rank routes its own tokens, sends each token-expert pair's x row to the
// rank owning the expert, the owners run their experts on the rows they
// received, the outputs travel back, and the source rank combines them with
// its router weights (section 专家混合模型) and applies the post-norm and the
// residual (section 残差流).
//
// Send order: the pairs in expert order (the permutation of the single-device
// path: by expert, stable by pair), so the rows for rank d -- experts
// [d E/P, (d+1) E/P) -- are one contiguous block.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_gemm.cuh"
#include "kernels_rows.cuh"

namespace beam {

constexpr int DEV_ERR_INDEX = 4;  // a caller-given expert index was outside [0, E) (pair dropped)

// Routing given by the caller, copied into the workspace: an index outside
// [0, E) raises the device error flag and the pair gets expert 0 with weight
// 0, so the layer completes without that contribution.
__global__ void __launch_bounds__(256) routed_copy_kernel(const int32_t* __restrict__ idx_in,
                                                          const float* __restrict__ w_in,
                                                          long long n, int E,
                                                          int32_t* __restrict__ idx_out,
                                                          float* __restrict__ w_out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int e = idx_in[i];
  const bool ok = e >= 0 && e < E;
  if (!ok) atomicOr(&g_beam_err, DEV_ERR_INDEX);
  idx_out[i] = ok ? e : 0;
  w_out[i] = ok ? w_in[i] : 0.f;
}

// Expert of every expert-ordered row (upper bound of the row in offsets[0..E])
// and the rows for each of the P ranks (experts per rank = E / P).
__global__ void __launch_bounds__(256) ep_meta_kernel(const int* __restrict__ offsets, int E, int P,
                                                      long long R, int32_t* __restrict__ row_expert,
                                                      int32_t* __restrict__ send_counts) {
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < R) {
    int lo = 0, hi = E - 1;   // last expert whose first row is <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
    }
    row_expert[r] = lo;
  }
  if (blockIdx.x == 0)
    for (int d = threadIdx.x; d < P; d += blockDim.x) {
      const int per = E / P;
      send_counts[d] = offsets[(d + 1) * per] - offsets[d * per];
    }
}

// Source-side combine of the returned expert outputs, then the output or the
// post-norm + scaled residual:
//   o[t,:] = sum_j w[t,j] * y[pair_row[t*k+j], :]   (FP32, slot order)
//   resid:  out = bf16( a * h_prev + b * RMSNorm(o) * gain )
//   else:   out = o  (bf16, or fp32 when OUT_F32)
// One block of 128 threads per token, 8 consecutive elements per thread and
// chunk, up to 8 chunks (H <= 8192).
constexpr int EP_COMBINE_THREADS = 128;

template <bool OUT_F32>
__global__ void __launch_bounds__(EP_COMBINE_THREADS) ep_combine_kernel(
    const float* __restrict__ y, const int32_t* __restrict__ pair_row,
    const float* __restrict__ topk_w, int top_k, const __nv_bfloat16* __restrict__ h_prev,
    const float* __restrict__ gain, void* __restrict__ out, int H, float eps, float a, float b,
    int resid) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  __shared__ float s_part[EP_COMBINE_THREADS / 32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < top_k) {
    s_row[tid] = pair_row[static_cast<size_t>(t) * top_k + tid];
    s_w[tid] = topk_w[static_cast<size_t>(t) * top_k + tid];
  }
  __syncthreads();
  const int nc = H >> 3;
  float o[8][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = tid + i * EP_COMBINE_THREADS;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[i][e] = 0.f;
    if (c >= nc) continue;
    for (int j = 0; j < top_k; ++j) {
      float f[8];
      load8(y + static_cast<size_t>(s_row[j]) * H, c, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[i][e] = fmaf(s_w[j], f[e], o[i][e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(o[i][e], o[i][e], ss);
  }
  float r = 1.f;
  if (resid) {
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < EP_COMBINE_THREADS / 32; ++w) tot += s_part[w];
    r = rsqrtf(tot / static_cast<float>(H) + eps);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = tid + i * EP_COMBINE_THREADS;
    if (c >= nc) continue;
    if (OUT_F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<size_t>(t) * H) + 2 * c;
      dst[0] = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
      dst[1] = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
      continue;
    }
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

}  // namespace beam
