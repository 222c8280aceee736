// Attention sublayer ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 注意力: grouped-query attention with 48 query and 8 key/value heads,
// RMSNorm on queries and keys, a sliding window of 512 tokens on most layers
// with RoPE, full context on every sixth layer and the last with the query
// scale (1 + (pos + 1) / 2048) ** 0.1 instead of positions, and a sigmoid
// gate from the layer input on every head channel before the output
// projection; section 残差流: RoPE and the query scaling in FP32). Head
// dimension 128 ("config.json" of the release, head_dim).
//
//   attn_prep_kernel       QK-RMSNorm, RoPE or query scale, gate sigmoid,
//                          from the FP32 fused projection
//   attn_vt_kernel         V transposed (keys contiguous)
//   linear_units_kernel    work list of a dense GEMM on the 2-SM pair kernel
//   flash_attn_kernel      softmax(Q K^T / sqrt(128) + mask) V per head on
//                          tcgen05 (S and O accumulate in TMEM), times the gate
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_gemm.cuh"
#include "kernels_permute.cuh"
#include "ptx.cuh"

namespace beam {

constexpr int ATT_D = 128;       // head dimension
constexpr int ATT_BQ = 128;      // query rows per CTA (the MMA's M)
constexpr int ATT_BK = 128;      // keys per tile (S's N, P V's K)

// ---------------------------------------------------------------------------
// prep: one warp per (token t, head slot s); slots [0, nq) query heads,
// [nq, nq+nkv) key heads, [nq+nkv, nq+2nkv) value heads, then nq gate heads.
// Lane l holds channels l, l+32, l+64, l+96, so the RoPE pairs (i, i+64) are
// in one lane. proj: [T, (2nq + 2nkv) * 128] FP32 (x W^T of the fused
// weight [W_q; W_k; W_v; W_g]).
//   q[h][t][:] = bf16(rope_or_scale(RMSNorm(q) * q_gain))   [nq][Tp][128]
//   k[g][t][:] = bf16(rope(RMSNorm(k) * k_gain))            [nkv][Tp][128]
//   gate[t][h*128 + c] = sigmoid(.)  (FP32)                 [T][nq*128]
// (value slots are written by attn_vt_kernel)
// window > 0: RoPE (theta) on q and k; window == 0: q *= (1 + (t+1)/2048)^0.1.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) attn_prep_kernel(
    const float* __restrict__ proj, int T, int Tp, int nq, int nkv,
    const float* __restrict__ q_gain, const float* __restrict__ k_gain, float eps, int window,
    float rope_theta, __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
    __nv_bfloat16* __restrict__ vt, float* __restrict__ gate) {
  const int t = blockIdx.x;
  const int slot = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nslots = 2 * nq + 2 * nkv;
  if (t >= T || slot >= nslots) return;
  const float* src = proj + static_cast<size_t>(t) * nslots * ATT_D + static_cast<size_t>(slot) * ATT_D;
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = src[lane + 32 * i];
  if (slot >= nq + 2 * nkv) {  // gate
    float* dst = gate + static_cast<size_t>(t) * nq * ATT_D + static_cast<size_t>(slot - nq - 2 * nkv) * ATT_D;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = 1.0f / (1.0f + expf(-v[i]));
    return;
  }
  if (slot >= nq + nkv) return;  // values: attn_vt_kernel
  const bool is_q = slot < nq;
  // RMSNorm over the head's 128 channels (FP32), gain per channel
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss / static_cast<float>(ATT_D) + eps);
  const float* gn = is_q ? q_gain : k_gain;
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= r * (gn ? gn[lane + 32 * i] : 1.f);
  if (window > 0) {
    // rotate-half RoPE: pairs (c, c + 64) for c = lane and lane + 32
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = lane + 32 * i;
      const float inv_freq = powf(rope_theta, -2.0f * static_cast<float>(c) / static_cast<float>(ATT_D));
      float sn, cs;
      sincosf(static_cast<float>(t) * inv_freq, &sn, &cs);
      const float x1 = v[i], x2 = v[i + 2];
      v[i] = x1 * cs - x2 * sn;
      v[i + 2] = x2 * cs + x1 * sn;
    }
  } else if (is_q) {
    const float s = powf(1.0f + (static_cast<float>(t) + 1.0f) / 2048.0f, 0.1f);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= s;
  }
  __nv_bfloat16* dst = is_q ? q + (static_cast<size_t>(slot) * Tp + t) * ATT_D
                            : k + (static_cast<size_t>(slot - nq) * Tp + t) * ATT_D;
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = __float2bfloat16_rn(v[i]);
}

// V transposed, keys contiguous: vt[g][c][t] = bf16(v[t][g][c]). One lane
// per token, a warp per 32 consecutive tokens of one key/value head, so the
// stores of a channel row are 64 contiguous bytes.
__global__ void __launch_bounds__(128) attn_vt_kernel(const float* __restrict__ proj, int T, int Tp,
                                                      int nq, int nkv,
                                                      __nv_bfloat16* __restrict__ vt) {
  const int t = blockIdx.x * 32 + (threadIdx.x & 31);
  const int g = blockIdx.y * 4 + (threadIdx.x >> 5);
  if (g >= nkv || t >= T) return;
  const int nslots = 2 * nq + 2 * nkv;
  const float4* src = reinterpret_cast<const float4*>(
      proj + static_cast<size_t>(t) * nslots * ATT_D + static_cast<size_t>(nq + nkv + g) * ATT_D);
  __nv_bfloat16* dst = vt + static_cast<size_t>(g) * ATT_D * Tp + t;
#pragma unroll 4
  for (int c4 = 0; c4 < ATT_D / 4; ++c4) {
    const float4 f = src[c4];
    dst[static_cast<size_t>(4 * c4) * Tp] = __float2bfloat16_rn(f.x);
    dst[static_cast<size_t>(4 * c4 + 1) * Tp] = __float2bfloat16_rn(f.y);
    dst[static_cast<size_t>(4 * c4 + 2) * Tp] = __float2bfloat16_rn(f.z);
    dst[static_cast<size_t>(4 * c4 + 3) * Tp] = __float2bfloat16_rn(f.w);
  }
}

// Work list of one dense GEMM (one "expert" of n rows) on the 2-SM pair
// kernel: units {0, first row, group size, weight tile} as pair_unit_at
// builds them for an expert; count in n_units[0].
__global__ void linear_units_kernel(int n, int MT, int4* __restrict__ units, int* __restrict__ n_units) {
  const int g = (n + 255) >> 8;
  const int total = MT * g;
  for (int l = blockIdx.x * blockDim.x + threadIdx.x; l < total; l += gridDim.x * blockDim.x)
    units[l] = pair_unit_at(l, 0, 0, n, MT);
  if (blockIdx.x == 0 && threadIdx.x == 0) n_units[0] = total;
}

// ---------------------------------------------------------------------------
// Flash attention on tcgen05, one CTA per (query tile of 128 rows, query
// head). Warp 0: TMA producer -- lane 0 loads Q once and then K tiles of 128
// keys into a three-stage ring (a stage is freed as soon as its S has been
// computed), lane 1 loads V^T tiles into a two-stage ring (freed after P V).
// Warp 1: TMEM owner and MMA issuer: S_0 and S_1 up front into two TMEM S
// buffers; then per tile j: O += P_j V_j as soon as P_j is ready, then
// S_{j+2} into the buffer S_j leaves. Warps 2..5 (thread = query row = TMEM
// lane): per tile read the S row, mask, online softmax in FP32 with a lazy
// reference: the row maximum m moves (and the O row in TMEM is rescaled)
// only when a tile's maximum exceeds m by more than ATT_TAU, so P <= e^TAU;
// the exponentials are computed before waiting for the previous P V; P is
// written as BF16 into the 128-byte-swizzled K-major tile the MMA reads. At
// the end O / l times the gate, BF16, to `out`.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384).
// All waits are bounded; on expiry the error word is set and every role
// leaves after its in-flight copies and MMAs have completed.
// ---------------------------------------------------------------------------
constexpr float ATT_TAU = 8.0f;

struct AttnArgs {
  int T, Tp, nq, nkv, window;
  float scale;                 // 1 / sqrt(head_dim)
  const float* gate;           // [T][nq * 128]
  __nv_bfloat16* out;          // [T][nq * 128]
  unsigned long long timeout_ns;
};

struct AttnCfg {
  static constexpr int Q_BYTES = ATT_BQ * ATT_D * 2;     // 32 KB: two 64-channel blocks
  static constexpr int K_BYTES = ATT_BK * ATT_D * 2;     // 32 KB
  static constexpr int V_BYTES = ATT_D * ATT_BK * 2;     // 32 KB (V^T: 128 channels x 128 keys)
  static constexpr int P_BYTES = ATT_BQ * ATT_BK * 2;    // 32 KB
  static constexpr int K_STAGES = 3, V_STAGES = 2;
  static constexpr int BAR_BYTES = 20 * 8 + 16;
  static constexpr int SMEM_BYTES =
      1024 + Q_BYTES + K_STAGES * K_BYTES + V_STAGES * V_BYTES + P_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// First and one-past-last key tile of query tile qt.
__device__ __forceinline__ void attn_key_tiles(int qt, int T, int window, int* j0, int* j1) {
  const int q0 = qt * ATT_BQ;
  const int qlast = min(q0 + ATT_BQ, T) - 1;
  const int kfirst = window > 0 ? max(0, q0 - window + 1) : 0;
  *j0 = kfirst / ATT_BK;
  *j1 = qlast / ATT_BK + 1;
}

__global__ void __launch_bounds__(192, 1)
    flash_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_vt, const AttnArgs args) {
  using C = AttnCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::Q_BYTES;
  uint8_t* sV = sK + C::K_STAGES * C::K_BYTES;
  uint8_t* sP = sV + C::V_STAGES * C::V_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + C::P_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;        // [3]
  uint64_t* k_empty = bars + 4;       // [3]
  uint64_t* v_full = bars + 7;        // [2]
  uint64_t* v_empty = bars + 9;       // [2]
  uint64_t* s_full = bars + 11;       // [2]
  uint64_t* p_full = bars + 13;
  uint64_t* o_done = bars + 14;
  uint64_t* mma_done = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heavy tiles first: the last query tiles of a causal global layer see the most keys
  const int qt = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y;
  const int g = h / (args.nq / args.nkv);
  int j0, j1;
  attn_key_tiles(qt, args.T, args.window, &j0, &j1);
  const int ntiles = j1 - j0;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::K_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::V_STAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producers
    if (lane < 2) {
      const uint64_t pol = l2_policy_evict_last();
      const volatile int never = 0;
      if (lane == 0) {
        const int qrow = h * args.Tp + qt * ATT_BQ;
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
        tma_load_2d(sQ, &tm_q, q_full, 0, qrow, pol);
        tma_load_2d(sQ + C::Q_BYTES / 2, &tm_q, q_full, 64, qrow, pol);
      }
      // lane 0: K tiles (3 stages); lane 1: V^T tiles (2 stages)
      const int NS = lane == 0 ? C::K_STAGES : C::V_STAGES;
      uint64_t* full = lane == 0 ? k_full : v_full;
      uint64_t* empty = lane == 0 ? k_empty : v_empty;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % NS;
        if (!mbar_wait_bounded(&empty[s], ((j / NS) & 1) ^ 1u, tmo, abort_flag)) {
          gemm_fail(abort_flag);
          break;
        }
        const int k0 = (j0 + j) * ATT_BK;
        mbar_arrive_expect_tx(&full[s], C::K_BYTES);
        if (lane == 0) {
          uint8_t* st = sK + s * C::K_BYTES;
          tma_load_2d(st, &tm_k, &full[s], 0, g * args.Tp + k0, pol);
          tma_load_2d(st + C::K_BYTES / 2, &tm_k, &full[s], 64, g * args.Tp + k0, pol);
        } else {
          uint8_t* st = sV + s * C::V_BYTES;
          tma_load_2d(st, &tm_vt, &full[s], k0, g * ATT_D, pol);
          tma_load_2d(st + C::V_BYTES / 2, &tm_vt, &full[s], k0 + 64, g * ATT_D, pol);
        }
        ++issued;
      }
      // every load must land before the CTA exits
      if (lane == 0 && !mbar_wait_bounded(q_full, 0, tmo, &never)) gemm_fail(abort_flag);
      for (int j = max(0, issued - NS); j < issued; ++j)
        if (!mbar_wait_bounded(&full[j % NS], (j / NS) & 1, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t dO = tmem_base + 256;
      bool ok = mbar_wait_bounded(q_full, 0, tmo, abort_flag);
      tc_fence_after();
      const uint64_t dq = sdesc_k128(smem_u32(sQ));
      const uint64_t dq1 = sdesc_k128(smem_u32(sQ + C::Q_BYTES / 2));
      const uint64_t dp = sdesc_k128(smem_u32(sP));
      const uint64_t dp1 = sdesc_k128(smem_u32(sP + C::P_BYTES / 2));
      auto issue_s = [&](int j) -> bool {
        const int ks = j % C::K_STAGES;
        if (!mbar_wait_bounded(&k_full[ks], (j / C::K_STAGES) & 1, tmo, abort_flag)) return false;
        tc_fence_after();
        const uint32_t base = smem_u32(sK + ks * C::K_BYTES);
        const uint64_t dk = sdesc_k128(base), dk1 = sdesc_k128(base + C::K_BYTES / 2);
        const uint32_t dS = tmem_base + static_cast<uint32_t>((j & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dS, dq + 2 * kk, dk + 2 * kk, idesc, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dS, dq1 + 2 * kk, dk1 + 2 * kk, idesc, 1u);
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[ks]);
        return true;
      };
      if (ok && ntiles > 0) ok = issue_s(0);
      if (ok && ntiles > 1) ok = issue_s(1);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int vs = j % C::V_STAGES;
        if (!mbar_wait_bounded(p_full, j & 1, tmo, abort_flag) ||
            !mbar_wait_bounded(&v_full[vs], (j / C::V_STAGES) & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(sV + vs * C::V_BYTES);
        const uint64_t dv = sdesc_k128(base), dv1 = sdesc_k128(base + C::V_BYTES / 2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, dp + 2 * kk, dv + 2 * kk, idesc, (j | kk) != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, dp1 + 2 * kk, dv1 + 2 * kk, idesc, 1u);
        mma_commit(o_done);
        mma_commit(&v_empty[vs]);
        // S_{j+2} into the buffer the softmax of tile j has finished reading
        if (j + 2 < ntiles && !issue_s(j + 2)) {
          ok = false;
          break;
        }
      }
      if (!ok) gemm_fail(abort_flag);
      mma_commit(mma_done);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                 // TMEM lane quarter
    const int row = q * 32 + lane;          // query row within the tile
    const int qi = qt * ATT_BQ + row;       // query index
    const uint32_t lanebits = static_cast<uint32_t>(q * 32) << 16;
    const float NEG = -1e30f;
    float m = NEG, l = 0.f;
    const float sc = args.scale;            // global layers' query scale is already in q
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      bool ready = false;
      if (lane == 0) ready = mbar_wait_bounded(&s_full[s], (j >> 1) & 1, tmo, abort_flag);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = (j0 + j) * ATT_BK;
      float sv[ATT_BK];
      tmem_ld128(tmem_base + lanebits + s * 128, sv);
      // visible keys: kj <= qi, kj < T and (window) qi - kj < window, i.e.
      // kj in [lo, hi]; reductions in eight independent partials (one warp per
      // scheduler: long dependency chains would stall it)
      const int hi = min(qi, args.T - 1);
      const int lo = args.window > 0 ? qi - args.window + 1 : 0;
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = NEG;
#pragma unroll
      for (int c = 0; c < ATT_BK; ++c) {
        const int kj = k0 + c;
        sv[c] = (kj >= lo && kj <= hi) ? sv[c] * sc : -INFINITY;
        mp[c & 7] = fmaxf(mp[c & 7], sv[c]);
      }
      const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      // lazy reference: move m only when this tile exceeds it by more than TAU
      const float mn = mt > m + ATT_TAU ? mt : m;
      const float alpha = __expf(m - mn);
      float sp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = 0.f;
#pragma unroll
      for (int c = 0; c < ATT_BK; ++c) {
        sv[c] = __expf(sv[c] - mn);
        sp[c & 7] += sv[c];
      }
      const float ps = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + ps;
      m = mn;
      // O may be rescaled and P overwritten only after the previous P V
      if (j > 0) {
        bool od = false;
        if (lane == 0) od = mbar_wait_bounded(o_done, (j - 1) & 1, tmo, abort_flag);
        od = __shfl_sync(0xffffffffu, od ? 1 : 0, 0) != 0;
        if (!od) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < ATT_D; c += 16) {
            float o[16];
            tmem_ld16(tmem_base + lanebits + 256 + c, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_st16(tmem_base + lanebits + 256 + c, o);
          }
          tmem_wait_st();
        }
      }
      // P row, BF16, into the swizzled K-major tile: key c of row `row` sits
      // in 64-key block c/64, 16-byte chunk (c%64)/8 ^ (row%8)
#pragma unroll
      for (int c8 = 0; c8 < ATT_BK / 8; ++c8) {
        uint4 pk;
        __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          p2[i] = __floats2bfloat162_rn(sv[c8 * 8 + 2 * i], sv[c8 * 8 + 2 * i + 1]);
        const int kb = c8 >> 3, chunk = c8 & 7;
        uint8_t* dst = sP + kb * (C::P_BYTES / 2) + (row >> 3) * 1024 + (row & 7) * 128 +
                       ((chunk ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = pk;
      }
      // P (generic-proxy stores) and the O rescale visible to the MMA
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // final: O / l times the gate, BF16
    bool od = ok;
    if (ok && ntiles > 0) {
      if (lane == 0) od = mbar_wait_bounded(o_done, (ntiles - 1) & 1, tmo, abort_flag);
      od = __shfl_sync(0xffffffffu, od ? 1 : 0, 0) != 0;
    }
    if (!od) {
      if (lane == 0) gemm_fail(abort_flag);
    } else {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool valid = qi < args.T;
      const size_t ld = static_cast<size_t>(args.nq) * ATT_D;
      const float* gr = args.gate + static_cast<size_t>(qi) * ld + static_cast<size_t>(h) * ATT_D;
      __nv_bfloat16* orow = args.out + static_cast<size_t>(qi) * ld + static_cast<size_t>(h) * ATT_D;
#pragma unroll 1
      for (int c = 0; c < ATT_D; c += 16) {
        float o[16];
        tmem_ld16(tmem_base + lanebits + 256 + c, o);
        if (valid) {
          float gt[16];
          const float4* g4 = reinterpret_cast<const float4*>(gr + c);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 t4 = g4[i];
            gt[4 * i] = t4.x; gt[4 * i + 1] = t4.y; gt[4 * i + 2] = t4.z; gt[4 * i + 3] = t4.w;
          }
          uint4 pk[2];
          __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            p2[i] = __floats2bfloat162_rn(o[2 * i] * inv_l * gt[2 * i], o[2 * i + 1] * inv_l * gt[2 * i + 1]);
          uint4* d4 = reinterpret_cast<uint4*>(orow + c);
          d4[0] = pk[0];
          d4[1] = pk[1];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace beam
