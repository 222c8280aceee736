// Router: FP32 logits, sigmoid scores, group-limited top-k and normalised
// weights.
//
// "Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文", section 专家混合模型:
// sigmoid scores over all experts; experts in groups of 32; keep the groups
// with the largest sum of their two best scores; top-8 experts inside the kept
// groups; weights normalised over the selected experts and multiplied by 2.5.
// Section 残差流: the router is computed in FP32.
// "Reflection 放出 501B 的 Beam 权重…", section "config.json 里还有六处能直接抄的细节":
// n_group 8, topk_group 4, norm_topk_prob, routed_scaling_factor 2.5.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace beam {

// ---------------------------------------------------------------------------
// logits partial sums: part[ks][t][e] = sum_{j in K-slice ks} x[t,j] * w[e,j]
// FP32 SIMT GEMM, 64 tokens x 64 experts per block, 4x4 outputs per thread,
// K-slices give enough blocks when T is small (decode).
// ---------------------------------------------------------------------------
constexpr int RL_BT = 64;
constexpr int RL_BE = 64;
constexpr int RL_BK = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ w,
                                                            float* __restrict__ part, int T,
                                                            int H, int E, int kslice) {
  __shared__ __align__(16) float xs[RL_BK][RL_BT + 4];
  __shared__ __align__(16) float ws[RL_BK][RL_BE + 4];
  const int t0 = blockIdx.x * RL_BT;
  const int e0 = blockIdx.y * RL_BE;
  const int ks = blockIdx.z;
  const int kbeg = ks * kslice;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const int lt = t0 + lr, le = e0 + lr;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = kbeg; k0 < kbeg + kslice; k0 += RL_BK) {
    {
      float f[8];
      if (lt < T) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(lt) * H + k0 + lk);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 q = __bfloat1622float2(p[i]);
          f[2 * i] = q.x;
          f[2 * i + 1] = q.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[lk + i][lr] = f[i];
    }
    {
      float f[8];
      if (le < E) {
        const float4* p = reinterpret_cast<const float4*>(w + static_cast<size_t>(le) * H + k0 + lk);
        const float4 a = p[0], b = p[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ws[lk + i][lr] = f[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RL_BK; ++kk) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
      const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int e = e0 + tx * 4;
  if (e < E) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + ty * 4 + i;
      if (t < T) {
        float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        *reinterpret_cast<float4*>(part + (static_cast<size_t>(ks) * T + t) * E + e) = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Exact three-way BF16 split of the FP32 router weight for the tensor-core
// logits GEMM: w = w1 + w2 + w3 with w1 = bf16(w), w2 = bf16(w - w1),
// w3 = bf16(w - w1 - w2) (each difference is exact in FP32). Output
// [E, 3H]: columns [0,H) hold w1, [H,2H) w2, [2H,3H) w3.
// ---------------------------------------------------------------------------
// Also writes the work list of the pair-kernel logits GEMM: units
// {K-split ks, first token, tokens (<= 256), 0}, split-major (the groups
// sharing a K-slice of the weight are adjacent), and their count.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ w, int E,
                                                           int H,
                                                           __nv_bfloat16* __restrict__ w3cat,
                                                           int T, int k_split,
                                                           int4* __restrict__ units,
                                                           int* __restrict__ n_units) {
  const int ngroups = (T + 255) / 256;
  if (blockIdx.x == 0) {
    for (int u = threadIdx.x; u < k_split * ngroups; u += blockDim.x) {
      const int ks = u / ngroups, j = u - ks * ngroups;
      units[u] = make_int4(ks, 256 * j, min(256, T - 256 * j), 0);
    }
    if (threadIdx.x == 0) *n_units = k_split * ngroups;
  }
  const size_t n = static_cast<size_t>(E) * H;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = i / H, j = i - e * H;
    const float v = w[i];
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(b);
    const __nv_bfloat16 c = __float2bfloat16_rn(r2);
    __nv_bfloat16* row = w3cat + e * 3 * H;
    row[j] = a;
    row[H + j] = b;
    row[2 * H + j] = c;
  }
}

// ---------------------------------------------------------------------------
// selection: one warp per token. Lane l holds experts e = 32*i + l for
// i < NI = E/32, so with groups of 32 experts group g is register column g and
// a group's top-2 is two warp max-reductions.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One block of 256 threads handles `tpb` (1..8) tokens: first all threads
// sum the K-slice partial logits of the block's (token, expert) pairs
// (coalesced over experts, slices summed in slice order) and apply bias and
// sigmoid into shared memory; then warp w selects for token tpb*blockIdx + w.
// Few tokens (many K-slices): one token per block, so the sums spread over
// many SMs; many tokens: 8 per block.
constexpr int SEL_TOKENS = 8;

template <int NI>
__global__ void __launch_bounds__(256) router_select_kernel(
    const float* __restrict__ part, int KS, const float* __restrict__ bias, int T, int E,
    int n_group, int topk_group, int top_k, float scale, int32_t* __restrict__ idx_out,
    float* __restrict__ w_out, float* __restrict__ scores_out, int tpb) {
  __shared__ float s_sc[SEL_TOKENS][NI * 32];
  const int t0 = blockIdx.x * tpb;
  for (int q = threadIdx.x; q < tpb * E; q += blockDim.x) {
    const int tl = q / E, e = q - tl * E;
    const int tt = t0 + tl;
    if (tt >= T) continue;
    const float* pk = part + static_cast<size_t>(tt) * E + e;
    const size_t kstride = static_cast<size_t>(T) * E;
    float l = 0.f;
#pragma unroll 8
    for (int k = 0; k < KS; ++k) l += pk[k * kstride];
    if (bias != nullptr) l += bias[e];
    const float sv = 1.0f / (1.0f + expf(-l));
    s_sc[tl][e] = sv;
    if (scores_out != nullptr) scores_out[static_cast<size_t>(tt) * E + e] = sv;
  }
  __syncthreads();
  const int t = t0 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) >= tpb || t >= T) return;

  float s[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) s[i] = s_sc[threadIdx.x >> 5][i * 32 + lane];

  // groups: keep topk_group of n_group (n_group == NI here unless all are kept)
  bool kept[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) kept[i] = true;
  if (topk_group < n_group) {
    float gs[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const float m1 = warp_max(s[i]);
      const unsigned at = __ballot_sync(0xffffffffu, s[i] == m1);
      const int first = __ffs(at) - 1;
      const float m2 = warp_max(lane == first ? -1.f : s[i]);
      gs[i] = m1 + m2;
      kept[i] = false;
    }
    for (int r = 0; r < topk_group; ++r) {
      float best = -2.f;
      int bi = 0;
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (!kept[i] && gs[i] > best) {
          best = gs[i];
          bi = i;
        }
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i == bi) kept[i] = true;
    }
  }

  // top_k among the kept experts: value descending, ties to the lower index
  float c[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) c[i] = kept[i] ? s[i] : -1.f;
  float my_s = 0.f, sum = 0.f;
  int my_e = 0;
  for (int j = 0; j < top_k; ++j) {
    float bv = -2.f;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (c[i] > bv) {
        bv = c[i];
        be = i * 32 + lane;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i == (be >> 5)) c[i] = -1.f;
    }
    if (lane == j) {
      my_s = bv;
      my_e = be;
    }
    sum += bv;
  }
  if (lane < top_k) {
    idx_out[static_cast<size_t>(t) * top_k + lane] = my_e;
    w_out[static_cast<size_t>(t) * top_k + lane] = scale * my_s / sum;
  }
}

}  // namespace beam
