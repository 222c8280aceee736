// Token -> expert permutation: per-block expert histograms, one scan that also
// builds the expert-GEMM work lists, a scatter that assigns every
// token-expert pair its row, and a gather that writes the expert-ordered copy
// of x. The pages only say that each token runs 8 of the
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

// Sum over the NB per-block histograms of expert e, and (second pass) the
// running offsets blk_off[b][e]; loads are issued eight at a time so their
// latencies overlap.
__device__ __forceinline__ int hist_total(const int* __restrict__ blk_hist, int NB, int E, int e) {
  int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int b = 0;
  for (; b + 8 <= NB; b += 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] += blk_hist[(b + j) * E + e];
  }
  for (; b < NB; ++b) acc[0] += blk_hist[b * E + e];
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}
__device__ __forceinline__ void hist_offsets(const int* __restrict__ blk_hist, int NB, int E,
                                             int e, int start, int* __restrict__ blk_off) {
  int run = start;
  int b = 0;
  for (; b + 8 <= NB; b += 8) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = blk_hist[(b + j) * E + e];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      blk_off[(b + j) * E + e] = run;
      run += v[j];
    }
  }
  for (; b < NB; ++b) {
    blk_off[b * E + e] = run;
    run += blk_hist[b * E + e];
  }
}

// Exclusive prefix sum over the 256 threads of a block; *total receives the
// sum of all values. s_warp holds 8 ints of scratch.
__device__ __forceinline__ int block_exclusive_scan256(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < 8 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < 8) s_warp[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? s_warp[warp - 1] : 0;
  *total = s_warp[7];
  __syncthreads();
  return base + x - v;
}

// One block of 256 threads (thread = expert, E <= 256).
//  counts[e], offsets[e] (exclusive scan, offsets[E] = T*top_k),
//  blk_off[b][e] = first row of block b's pairs of expert e,
//  and the token-tile list of the weight-major GEMMs: tiles[k] = {expert,
//  first row, rows (<= NT), 0}, experts ordered by token count (descending,
//  ties to the lower index). The GEMMs expand unit u into tile u / MT and
//  weight row-tile u % MT, so a few hundred tiles describe all units.
//  n_units = {tiles * MT_gu, tiles * MT_dn, tiles, 0}.
// With pad > 1 every expert's rows start at a multiple of `pad` (its row
// range is padded to a multiple of pad; offsets[E] is the padded total) and
// the padding rows get row_token = -1.
__global__ void __launch_bounds__(256) expert_scan_units_kernel(
    const int* __restrict__ blk_hist, int NB, int E, int* __restrict__ blk_off,
    int* __restrict__ counts, int* __restrict__ offsets, int4* __restrict__ tiles,
    int* __restrict__ n_units, int NT, int MT_gu, int MT_dn, int pad,
    int* __restrict__ row_token) {
  __shared__ int s_cnt[256];
  __shared__ int s_off[256];
  __shared__ int s_order[256];
  __shared__ int s_warp[8];
  const int e = threadIdx.x;
  const int c = e < E ? hist_total(blk_hist, NB, E, e) : 0;
  s_cnt[e] = (e < E) ? c : 0;
  int total = 0;
  const int cpad = (c + pad - 1) / pad * pad;
  const int off = block_exclusive_scan256(e < E ? cpad : 0, s_warp, &total);
  s_off[e] = off;
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    if (e == 0) offsets[E] = total;
    hist_offsets(blk_hist, NB, E, e, off, blk_off);
    for (int r = off + c; r < off + cpad; ++r) row_token[r] = -1;
    int rank = 0;
    for (int j = 0; j < E; ++j) rank += (s_cnt[j] > c) || (s_cnt[j] == c && j < e);
    s_order[rank] = e;
  }
  __syncthreads();
  const int ex = e < E ? s_order[e] : 0;
  const int n = e < E ? s_cnt[ex] : 0;
  const int nt = (n + NT - 1) / NT;
  int ntiles = 0;
  const int tb = block_exclusive_scan256(nt, s_warp, &ntiles);
  if (e == 0) {
    n_units[0] = ntiles * MT_gu;
    n_units[1] = ntiles * MT_dn;
    n_units[2] = ntiles;
    n_units[3] = 0;
  }
  const int r0 = s_off[ex];
  for (int j = 0; j < nt; ++j) tiles[tb + j] = make_int4(ex, r0 + j * NT, min(NT, n - j * NT), 0);
}

// Work lists of the token-major two-CTA GEMMs. A cluster unit is two int4
// sub-units, one per CTA: {expert, first row, rows (<= 128), weight tile |
// TM_PAIR}. An expert's rows go in 256-row groups, each a PAIR unit (both
// CTAs on the same weight tile, 128 rows each); a last
// remainder of at most 128 rows becomes SOLO sub-units -- one per weight
// tile, two tiles per cluster unit, each CTA loading its own weights -- so a
// tail costs one 128-row MMA tile instead of a 256-row group. Units of one
// expert are contiguous, tiles in ascending order; experts by token count,
// descending. A sub-unit with 0 rows repeats a valid tile and stores nothing.
constexpr int TM_PAIR = 0x40000000;

__device__ __forceinline__ int tm_units_for(int n, int MT) {
  const int q = n >> 8, rem = n & 255;
  const int pairs = q + (rem > 128 ? 1 : 0);
  const int tail = (rem > 0 && rem <= 128) ? 1 : 0;
  return MT * pairs + tail * ((MT + 1) >> 1);
}

// Unit l (0-based, within one expert's contiguous run) of each list format,
// computed directly, so all threads of a block can write any expert's units.
// tm: per pair of weight tiles (m, m+1): `pairs` PAIR units for m, `pairs`
// for m+1, then one SOLO unit for the tail (when there is one); a last odd
// tile has `pairs` PAIR units and the tail.
__device__ __forceinline__ void tm_unit_at(int l, int ex, int r0, int n, int MT, int4* out2) {
  const int q = n >> 8, rem = n & 255;
  const int pairs = q + (rem > 128 ? 1 : 0);
  const int tail = (rem > 0 && rem <= 128) ? rem : 0;
  const int per = 2 * pairs + (tail ? 1 : 0);
  const int nfull = MT >> 1;
  int b, r, mm;
  if (l < nfull * per) {
    b = l / per;
    r = l - b * per;
    mm = 2;
  } else {
    b = nfull;
    r = l - nfull * per;
    mm = 1;
  }
  const int m = 2 * b;
  if (r < pairs * mm) {
    const int mo = r / pairs, g = r - mo * pairs;
    const int gr = r0 + 256 * g, gn = n - 256 * g;
    out2[0] = make_int4(ex, gr, min(128, gn), (m + mo) | TM_PAIR);
    out2[1] = make_int4(ex, gr + 128, max(0, min(128, gn - 128)), (m + mo) | TM_PAIR);
  } else {
    const int tr = r0 + 256 * q;
    out2[0] = make_int4(ex, tr, tail, m);
    out2[1] = (m + 1 < MT) ? make_int4(ex, tr, tail, m + 1) : make_int4(ex, tr, 0, m);
  }
}

// pair (2-SM) lists: an expert's n tokens are split into g = ceil(n / 256)
// balanced groups; a unit is {expert, first row, group size, weight tile},
// weight-tile-major (the groups sharing a tile are adjacent): unit l is
// weight tile m = l / g, group l % g.
__device__ __forceinline__ int4 pair_unit_at(int l, int ex, int r0, int n, int MT) {
  const int g = (n + 255) >> 8;
  const int q = n / g, extra = n - q * g;
  const int m = l / g, gi = l - m * g;
  const int start = gi * q + min(gi, extra);
  return make_int4(ex, r0 + start, q + (gi < extra ? 1 : 0), m);
}

// Work lists for prefill: each GEMM's list in the format of the kernel that
// runs it (LIST_TM: two-CTA token-major cluster units; LIST_PAIR: 2-SM pair
// units of the wide kernel, MT weight slices per expert). Also writes
// counts, offsets and the per-block row offsets.
constexpr int LIST_TM = 0;
constexpr int LIST_PAIR = 1;

template <int KIND>
__device__ __forceinline__ int list_units_for(int n, int MT) {
  return KIND == LIST_TM ? tm_units_for(n, MT) : ((n + 255) >> 8) * MT;
}
// Unit u of a list = unit l of expert run (ex, r0, n).
template <int KIND>
__device__ __forceinline__ void list_unit(int4* units, int u, int l, int ex, int r0, int n, int MT) {
  if (KIND == LIST_TM) {
    int4 two[2];
    tm_unit_at(l, ex, r0, n, MT, two);
    units[2 * u] = two[0];
    units[2 * u + 1] = two[1];
  } else {
    units[u] = pair_unit_at(l, ex, r0, n, MT);
  }
}

template <int GU_KIND, int DN_KIND>
__global__ void __launch_bounds__(256) expert_scan_units_prefill_kernel(
    const int* __restrict__ blk_hist, int NB, int E, int* __restrict__ blk_off,
    int* __restrict__ counts, int* __restrict__ offsets, int4* __restrict__ units_gu,
    int4* __restrict__ units_dn, int* __restrict__ n_units, int MT_gu, int MT_dn, int pad = 1,
    int* __restrict__ row_token = nullptr) {
  __shared__ int s_cnt[256];
  __shared__ int s_pad[256];
  __shared__ int s_order[256];
  __shared__ int s_warp[8];
  const int e = threadIdx.x;
  const int c = e < E ? hist_total(blk_hist, NB, E, e) : 0;
  s_cnt[e] = (e < E) ? c : 0;
  // pad > 1: every expert's rows start at a multiple of pad; the padding rows
  // get row_token = -1
  const int cpad = (c + pad - 1) / pad * pad;
  s_pad[e] = (e < E) ? cpad : 0;
  int total = 0;
  const int off = block_exclusive_scan256(e < E ? cpad : 0, s_warp, &total);
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    if (e == 0) offsets[E] = total;
    hist_offsets(blk_hist, NB, E, e, off, blk_off);
    if (pad > 1)
      for (int r = off + c; r < off + cpad; ++r) row_token[r] = -1;
    int rank = 0;
    for (int j = 0; j < E; ++j) rank += (s_cnt[j] > c) || (s_cnt[j] == c && j < e);
    s_order[rank] = e;
  }
  __syncthreads();
  const int ex = e < E ? s_order[e] : 0;
  const int n = e < E ? s_cnt[ex] : 0;
  int r0 = 0;
  for (int j = 0; j < ex; ++j) r0 += s_pad[j];
  int tot_gu = 0, tot_dn = 0;
  const int b_gu = block_exclusive_scan256(n > 0 ? list_units_for<GU_KIND>(n, MT_gu) : 0, s_warp,
                                           &tot_gu);
  const int b_dn = block_exclusive_scan256(n > 0 ? list_units_for<DN_KIND>(n, MT_dn) : 0, s_warp,
                                           &tot_dn);
  if (e == 0) {
    n_units[0] = tot_gu;
    n_units[1] = tot_dn;
    n_units[2] = 0;
    n_units[3] = 0;
  }
  // Cooperative writes: unit u belongs to the sorted position p whose base is
  // the largest <= u (binary search over the bases in shared memory).
  __shared__ int s_bgu[257], s_bdn[257], s_ex[256], s_r0[256], s_n[256];
  s_bgu[e] = b_gu;
  s_bdn[e] = b_dn;
  s_ex[e] = ex;
  s_r0[e] = r0;
  s_n[e] = n;
  if (e == 0) {
    s_bgu[256] = tot_gu;
    s_bdn[256] = tot_dn;
  }
  __syncthreads();
  for (int u = e; u < tot_gu; u += blockDim.x) {
    int lo = 0, hi = 255;  // last position with base <= u (positions with 0 units share bases)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_bgu[mid] <= u) lo = mid; else hi = mid - 1;
    }
    list_unit<GU_KIND>(units_gu, u, u - s_bgu[lo], s_ex[lo], s_r0[lo], s_n[lo], MT_gu);
  }
  for (int u = e; u < tot_dn; u += blockDim.x) {
    int lo = 0, hi = 255;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_bdn[mid] <= u) lo = mid; else hi = mid - 1;
    }
    list_unit<DN_KIND>(units_dn, u, u - s_bdn[lo], s_ex[lo], s_r0[lo], s_n[lo], MT_dn);
  }
}

// At most PERM_TPB tokens (one permutation block): the histogram, the scan
// with the token-tile work list and the scatter of expert_block_hist_kernel,
// expert_scan_units_kernel and expert_scatter_kernel in one launch of one
// block of 256 threads, with the same outputs (blk_hist / blk_off are not
// needed and not written).
__global__ void __launch_bounds__(256) expert_permute_small_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, int T, int top_k, int E,
    int* __restrict__ counts, int* __restrict__ offsets, int4* __restrict__ tiles,
    int* __restrict__ n_units, int NT, int MT_gu, int MT_dn, int pad,
    int* __restrict__ pair_row, int* __restrict__ row_token, float* __restrict__ row_weight) {
  __shared__ int s_e[PERM_TPB * 32];
  __shared__ int s_cnt[256];
  __shared__ int s_off[256];
  __shared__ int s_order[256];
  __shared__ int s_warp[8];
  const int e = threadIdx.x;
  const int np = T * top_k;
  s_cnt[e] = 0;
  __syncthreads();
  for (int p = e; p < np; p += blockDim.x) {
    const int x = idx[p];
    s_e[p] = x;
    atomicAdd(&s_cnt[x], 1);
  }
  __syncthreads();
  const int c = s_cnt[e];                 // 0 for e >= E
  int total = 0;
  const int cpad = (c + pad - 1) / pad * pad;
  const int off = block_exclusive_scan256(e < E ? cpad : 0, s_warp, &total);
  s_off[e] = off;
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    if (e == 0) offsets[E] = total;
    for (int r = off + c; r < off + cpad; ++r) row_token[r] = -1;
    int rank = 0;
    for (int j = 0; j < E; ++j) rank += (s_cnt[j] > c) || (s_cnt[j] == c && j < e);
    s_order[rank] = e;
  }
  __syncthreads();
  // token-tile work list, experts by token count (descending, ties to the
  // lower index)
  const int ex = e < E ? s_order[e] : 0;
  const int n = e < E ? s_cnt[ex] : 0;
  const int nt = (n + NT - 1) / NT;
  int ntiles = 0;
  const int tb = block_exclusive_scan256(nt, s_warp, &ntiles);
  if (e == 0) {
    n_units[0] = ntiles * MT_gu;
    n_units[1] = ntiles * MT_dn;
    n_units[2] = ntiles;
    n_units[3] = 0;
  }
  const int r0 = s_off[ex];
  for (int j = 0; j < nt; ++j) tiles[tb + j] = make_int4(ex, r0 + j * NT, min(NT, n - j * NT), 0);
  // pair p's row: its expert's first row plus its stable rank among the
  // expert's pairs
  for (int p = e; p < np; p += blockDim.x) {
    const int x = s_e[p];
    int r = 0;
    for (int q = 0; q < p; ++q) r += (s_e[q] == x);
    const int row = s_off[x] + r;
    pair_row[p] = row;
    row_token[row] = p / top_k;
    row_weight[row] = wts[p];
  }
}

// Row of every pair of this block in the expert-ordered layout: pair_row[p],
// and the inverse maps row_token / row_weight.
__global__ void __launch_bounds__(PERM_THREADS) expert_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, int T, int top_k, int E,
    const int* __restrict__ blk_off, int* __restrict__ pair_row, int* __restrict__ row_token,
    float* __restrict__ row_weight) {
  __shared__ int s_e[PERM_TPB * 32];
  const int p0 = blockIdx.x * PERM_TPB * top_k;
  const int np = min(PERM_TPB * top_k, T * top_k - p0);
  for (int p = threadIdx.x; p < np; p += blockDim.x) s_e[p] = idx[p0 + p];
  __syncthreads();
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const int e = s_e[p];
    int r = 0;
    for (int q = 0; q < p; ++q) r += (s_e[q] == e);
    const int row = blk_off[blockIdx.x * E + e] + r;
    pair_row[p0 + p] = row;
    row_token[row] = (p0 + p) / top_k;
    row_weight[row] = wts[p0 + p];
  }
}

// Identity routing for the dense SwiGLU MLP (one expert that every token uses
// with weight 1): the histogram of the single block and the maps.
__global__ void __launch_bounds__(256) dense_setup_kernel(int T, int* __restrict__ blk_hist,
                                                          int* __restrict__ pair_row,
                                                          int* __restrict__ row_token,
                                                          float* __restrict__ row_weight,
                                                          float* __restrict__ w) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) blk_hist[0] = T;
  if (t < T) {
    pair_row[t] = t;
    row_token[t] = t;
    row_weight[t] = 1.f;
    w[t] = 1.f;
  }
}

// xperm[row, :] = x[row_token[row], :], one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int* __restrict__ row_token,
                                                          int R, int H,
                                                          __nv_bfloat16* __restrict__ xperm) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  const int t = row_token[row];
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  uint4* dst = reinterpret_cast<uint4*>(xperm + static_cast<size_t>(row) * H);
  const int nc = H >> 3;
  for (int c = lane; c < nc; c += 32) dst[c] = src[c];
}

}  // namespace beam
