// Attention sublayer ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 注意力: grouped-query attention with 48 query and 8 key/value heads,
// RMSNorm on queries and keys, a sliding window of 512 tokens on most layers
// with RoPE, full context on every sixth layer and the last with the query
// scale (1 + (pos + 1) / 2048) ** 0.1 instead of positions, and a sigmoid
// gate from the layer input on every head channel before the output
// projection; section 残差流: RoPE and the query scaling in FP32). Head
// dimension 128 ("config.json" of the release, head_dim).
//
//   attn_prep_kernel       QK-RMSNorm, RoPE or query scale, V transposed,
//                          gate sigmoid, from the FP32 fused projection
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
//   vt[g][c][t] = bf16(v[t][g][c])                          [nkv][128][Tp]
//   gate[t][h*128 + c] = sigmoid(.)  (FP32)                 [T][nq*128]
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
  if (slot >= nq + nkv) {      // value: transposed, keys contiguous
    const int g = slot - nq - nkv;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      vt[(static_cast<size_t>(g) * ATT_D + lane + 32 * i) * Tp + t] = __float2bfloat16_rn(v[i]);
    return;
  }
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
// head). Warp 0: TMA producer (Q once, then K and V^T tiles of 128 keys into
// a two-stage ring). Warp 1: TMEM owner and MMA issuer: S_j = Q K_j^T into
// one of two TMEM S buffers, then O += P_j V_j into TMEM once P_j is ready.
// Warps 2..5 (thread = query row = TMEM lane): per tile read S, mask, online
// softmax in FP32 (running max m and sum l), rescale the O row in TMEM when
// m grows, write P (BF16) into shared memory in the MMA's 128-byte-swizzled
// K-major layout; at the end O / l times the gate, BF16, to `out`.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384).
// All waits are bounded; on expiry the error word is set and every role
// leaves after in-flight copies and MMAs have completed.
// ---------------------------------------------------------------------------
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
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  static constexpr int BAR_BYTES = 16 * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + Q_BYTES + 2 * STAGE_BYTES + P_BYTES + BAR_BYTES;
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
  uint8_t* sKV = sQ + C::Q_BYTES;                    // stage s: K at s*STAGE, V^T after
  uint8_t* sP = sKV + 2 * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + C::P_BYTES);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;       // [2]
  uint64_t* kv_empty = bars + 3;      // [2]
  uint64_t* s_full = bars + 5;        // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* o_done = bars + 8;
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      const int qrow = h * args.Tp + qt * ATT_BQ;
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      tma_load_2d(sQ, &tm_q, q_full, 0, qrow, pol);
      tma_load_2d(sQ + C::Q_BYTES / 2, &tm_q, q_full, 64, qrow, pol);
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j & 1;
        if (!mbar_wait_bounded(&kv_empty[s], ((j >> 1) & 1) ^ 1u, tmo, abort_flag)) {
          gemm_fail(abort_flag);
          break;
        }
        uint8_t* st = sKV + s * C::STAGE_BYTES;
        const int k0 = (j0 + j) * ATT_BK;
        mbar_arrive_expect_tx(&kv_full[s], C::STAGE_BYTES);
        tma_load_2d(st, &tm_k, &kv_full[s], 0, g * args.Tp + k0, pol);
        tma_load_2d(st + C::K_BYTES / 2, &tm_k, &kv_full[s], 64, g * args.Tp + k0, pol);
        tma_load_2d(st + C::K_BYTES, &tm_vt, &kv_full[s], k0, g * ATT_D, pol);
        tma_load_2d(st + C::K_BYTES + C::V_BYTES / 2, &tm_vt, &kv_full[s], k0 + 64, g * ATT_D, pol);
        ++issued;
      }
      // every load must land before the CTA exits
      const volatile int never = 0;
      if (!mbar_wait_bounded(q_full, 0, tmo, &never)) gemm_fail(abort_flag);
      for (int j = issued - 2; j < issued; ++j)
        if (j >= 0 && !mbar_wait_bounded(&kv_full[j & 1], (j >> 1) & 1, tmo, &never))
          gemm_fail(abort_flag);
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
        const int s = j & 1;
        if (!mbar_wait_bounded(&kv_full[s], (j >> 1) & 1, tmo, abort_flag)) return false;
        tc_fence_after();
        const uint32_t base = smem_u32(sKV + s * C::STAGE_BYTES);
        const uint64_t dk = sdesc_k128(base), dk1 = sdesc_k128(base + C::K_BYTES / 2);
        const uint32_t dS = tmem_base + static_cast<uint32_t>(s * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dS, dq + 2 * kk, dk + 2 * kk, idesc, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dS, dq1 + 2 * kk, dk1 + 2 * kk, idesc, 1u);
        mma_commit(&s_full[s]);
        return true;
      };
      if (ok && ntiles > 0) ok = issue_s(0);
      for (int j = 0; ok && j < ntiles; ++j) {
        // S_{j+1} overlaps the softmax of tile j (its buffer was read by the
        // softmax of tile j-1, which signalled p_full before this point)
        if (j + 1 < ntiles && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(p_full, j & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(sKV + (j & 1) * C::STAGE_BYTES);
        const uint64_t dv = sdesc_k128(base + C::K_BYTES), dv1 = sdesc_k128(base + C::K_BYTES + C::V_BYTES / 2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, dp + 2 * kk, dv + 2 * kk, idesc, (j | kk) != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss(dO, dp1 + 2 * kk, dv1 + 2 * kk, idesc, 1u);
        mma_commit(o_done);
        mma_commit(&kv_empty[j & 1]);
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
    // softmax scale; global layers' query scale is already in q
    const float sc = args.scale;
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
#pragma unroll
      for (int c = 0; c < ATT_BK; c += 32) {
        float a[16], b[16];
        tmem_ld16x2(tmem_base + lanebits + s * 128 + c, tmem_base + lanebits + s * 128 + c + 16, a, b);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sv[c + i] = a[i];
          sv[c + 16 + i] = b[i];
        }
      }
      float mt = NEG;
#pragma unroll
      for (int c = 0; c < ATT_BK; ++c) {
        const int kj = k0 + c;
        const bool vis = kj <= qi && kj < args.T && (args.window == 0 || qi - kj < args.window);
        sv[c] = vis ? sv[c] * sc : -INFINITY;
        mt = fmaxf(mt, sv[c]);
      }
      const float mn = fmaxf(m, mt);
      const float alpha = __expf(m - mn);
      // the O row may be rescaled only after the previous P V has completed
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
      float ps = 0.f;
      // P row, BF16, into the swizzled K-major tile: key c of row `row` sits
      // in 64-key block c/64, 16-byte chunk (c%64)/8 ^ (row%8)
#pragma unroll
      for (int c8 = 0; c8 < ATT_BK / 8; ++c8) {
        float p8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p8[i] = __expf(sv[c8 * 8 + i] - mn);
          ps += p8[i];
        }
        uint4 pk;
        __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) p2[i] = __floats2bfloat162_rn(p8[2 * i], p8[2 * i + 1]);
        const int kb = c8 >> 3, chunk = c8 & 7;
        uint8_t* dst = sP + kb * (C::P_BYTES / 2) + (row >> 3) * 1024 + (row & 7) * 128 +
                       ((chunk ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = pk;
      }
      l = l * alpha + ps;
      m = mn;
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
          uint4 pk[2];
          __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            p2[i] = __floats2bfloat162_rn(o[2 * i] * inv_l * gr[c + 2 * i], o[2 * i + 1] * inv_l * gr[c + 2 * i + 1]);
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
