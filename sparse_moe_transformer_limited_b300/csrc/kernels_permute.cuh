// Token -> expert permutation: per-block expert histograms, one scan that also
// builds the expert-GEMM work lists, and a scatter that writes the
// expert-ordered copy of x. The pages only say that each token runs 8 of the
// 256 experts ("Reflection 发布 Beam 501B 开源模型…", section 专家混合模型); grouping
// the token-expert pairs by expert is what lets each expert's weights stream
// once per token tile.
//
// Pair p = t * top_k + j (token t, slot j). Rows of the expert-ordered layout
// are sorted by expert and, inside an expert, by pair index (stable).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace beam {

constexpr int PERM_TPB = 64;       // tokens per permutation block
constexpr int PERM_THREADS = 512;

// blk_hist[b][e] = number of pairs of block b routed to expert e
__global__ void __launch_bounds__(PERM_THREADS) expert_block_hist_kernel(
    const int32_t* __restrict__ idx, int T, int top_k, int E, int* __restrict__ blk_hist) {
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * PERM_TPB * top_k;
  const int np = min(PERM_TPB * top_k, T * top_k - p0);
  for (int p = threadIdx.x; p < np; p += blockDim.x) atomicAdd(&hist[idx[p0 + p]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_hist[blockIdx.x * E + e] = hist[e];
}

// One block of 256 threads (thread = expert, E <= 256).
//  counts[e], offsets[e] (exclusive scan, offsets[E] = T*top_k),
//  blk_off[b][e] = first row of block b's pairs of expert e,
//  work lists for the two expert GEMMs. A unit is int4 {expert, first row,
//  rows (<= NT), weight row-tile}. Experts are ordered by token count
//  (descending, ties to the lower index); inside an expert, units run
//  row-tile-major so the token tiles sharing one weight tile are adjacent.
__global__ void __launch_bounds__(256) expert_scan_units_kernel(
    const int* __restrict__ blk_hist, int NB, int E, int* __restrict__ blk_off,
    int* __restrict__ counts, int* __restrict__ offsets, int4* __restrict__ units_gu,
    int4* __restrict__ units_dn, int* __restrict__ n_units, int NT, int MT_gu, int MT_dn) {
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  __shared__ int s_order[256];
  __shared__ int s_tbase[257];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int b = 0; b < NB; ++b) c += blk_hist[b * E + e];
  s_cnt[e] = (e < E) ? c : 0;
  __syncthreads();
  if (e == 0) {
    int run = 0;
    for (int i = 0; i < E; ++i) {
      s_off[i] = run;
      run += s_cnt[i];
    }
    s_off[E] = run;
  }
  __syncthreads();
  if (e < E) {
    counts[e] = s_cnt[e];
    offsets[e] = s_off[e];
    if (e == 0) offsets[E] = s_off[E];
    int run = s_off[e];
    for (int b = 0; b < NB; ++b) {
      blk_off[b * E + e] = run;
      run += blk_hist[b * E + e];
    }
    int rank = 0;
    const int me = s_cnt[e];
    for (int j = 0; j < E; ++j) rank += (s_cnt[j] > me) || (s_cnt[j] == me && j < e);
    s_order[rank] = e;
  }
  __syncthreads();
  if (e == 0) {
    int run = 0;
    for (int p = 0; p < E; ++p) {
      s_tbase[p] = run;
      run += (s_cnt[s_order[p]] + NT - 1) / NT;
    }
    s_tbase[E] = run;
    n_units[0] = run * MT_gu;
    n_units[1] = run * MT_dn;
    n_units[2] = run;
    n_units[3] = 0;
  }
  __syncthreads();
  if (e < E) {
    const int ex = s_order[e];
    const int n = s_cnt[ex];
    const int nt = (n + NT - 1) / NT;
    const int tb = s_tbase[e];
    const int r0 = s_off[ex];
    for (int m = 0; m < MT_gu; ++m)
      for (int j = 0; j < nt; ++j)
        units_gu[static_cast<size_t>(tb) * MT_gu + m * nt + j] =
            make_int4(ex, r0 + j * NT, min(NT, n - j * NT), m);
    for (int m = 0; m < MT_dn; ++m)
      for (int j = 0; j < nt; ++j)
        units_dn[static_cast<size_t>(tb) * MT_dn + m * nt + j] =
            make_int4(ex, r0 + j * NT, min(NT, n - j * NT), m);
  }
}

// Rows of this block's pairs, row_token / row_weight, and the expert-ordered
// copy of x (one warp copies one row with 16-byte loads and stores).
__global__ void __launch_bounds__(PERM_THREADS) expert_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, int T, int top_k, int E,
    const int* __restrict__ blk_off, const __nv_bfloat16* __restrict__ x, int H,
    int* __restrict__ row_token, float* __restrict__ row_weight,
    __nv_bfloat16* __restrict__ xperm) {
  extern __shared__ int sm[];
  int* s_e = sm;
  int* s_row = sm + PERM_TPB * top_k;
  const int p0 = blockIdx.x * PERM_TPB * top_k;
  const int np = min(PERM_TPB * top_k, T * top_k - p0);
  for (int p = threadIdx.x; p < np; p += blockDim.x) s_e[p] = idx[p0 + p];
  __syncthreads();
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const int e = s_e[p];
    int r = 0;
    for (int q = 0; q < p; ++q) r += (s_e[q] == e);
    const int row = blk_off[blockIdx.x * E + e] + r;
    s_row[p] = row;
    row_token[row] = (p0 + p) / top_k;
    row_weight[row] = wts[p0 + p];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int nc = H >> 3;
  for (int p = warp; p < np; p += nw) {
    const int t = (p0 + p) / top_k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(xperm + static_cast<size_t>(s_row[p]) * H);
    for (int c = lane; c < nc; c += 32) dst[c] = src[c];
  }
}

}  // namespace beam
