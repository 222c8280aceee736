// Token-major gate/up expert GEMM with 256 token rows per CTA (prefill), on
// tcgen05 + TMEM, one CTA per SM, no cluster.
//
// The layer's experts ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 专家混合模型): SwiGLU MLPs, hidden 5120, intermediate 2560, the
// SwiGLU product in FP32 (section 残差流).
//
// A unit is (expert e, weight tile n, up to 256 consecutive rows of e in the
// expert-ordered token layout). Per K-block the stage holds the unit's token
// rows as two 128-row halves (A0, A1) and one 256-row weight tile B = [W_g
// rows 128n .. 128n+127 ; W_u rows 128n .. 128n+127]; two M = 128, N = 256
// MMAs (one per half) read the same B. Against the two-CTA multicast kernel
// (128 rows per CTA, B filled half by TMA and half by the peer's multicast)
// every weight byte written into shared memory now feeds two MMAs, so per
// 256 x 256 x 64 step an SM moves 64 KB in by TMA and 96 KB out to the tensor
// core instead of 2 x 96 KB -- shared memory, not the tensor core, binds
// these GEMMs. A unit of at most 128 rows runs the first half only.
//
// TMEM: accumulator of half 0 in columns [0, 256) (gate 0..127, up
// 128..255), half 1 in [256, 512); one accumulator pair, so the epilogue of a
// unit must drain before the next unit's first MMA. Epilogue: 8 warps, warp
// (lane quarter q = warp % 4, half h) owns 32 rows of half h and writes
// act[row, 128n + i] = bf16(silu(g_i) * u_i) in FP32, 32 columns at a time.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps
// 2..9 epilogue. All waits are bounded.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_gemm.cuh"
#include "kernels_permute.cuh"
#include "ptx.cuh"

namespace beam {

struct Tm2Args {
  const int4* units;        // {expert, first row, rows (1..256), weight tile}
  const int* n_units;
  int k_blocks;             // 128-byte K-blocks: K / 64 (BF16) or K / 128 (E4M3)
  int w_rows_per_expert;    // I
  __nv_bfloat16* out;       // act [R, I] bf16
  int out_ld;
  unsigned long long timeout_ns;
  // E4M3 operands only: per token-row scale and per weight-row scales of the
  // gate and up matrices, indexed expert * I + row
  const float* row_scale;
  const float* w_scale0;
  const float* w_scale1;
};

template <int KIND>
struct Tm2Cfg {
  static constexpr int HALF_A = 128 * 128;                // 16 KB: 128 token rows x 128 bytes
  static constexpr int A_BYTES = 2 * HALF_A;
  static constexpr int B_BYTES = 256 * 128;               // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 64 KB
  static constexpr int STAGES = 3;
  static constexpr int TMEM_COLS = 512;
  static constexpr int BAR_BYTES = (2 * STAGES + 3) * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

constexpr int TM2_THREADS = 320;

template <int KIND>
__global__ void __launch_bounds__(TM2_THREADS, 1)
    expert_gemm_tm2_kernel(const __grid_constant__ CUtensorMap tm_wg,
                           const __grid_constant__ CUtensorMap tm_wu,
                           const __grid_constant__ CUtensorMap tm_tok, const Tm2Args args) {
  using C = Tm2Cfg<KIND>;
  constexpr bool F8 = KIND == KIND_E4M3;
  static_assert(KIND == KIND_BF16 || KIND == KIND_E4M3, "BF16 or E4M3 operands");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* mma_done = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 8);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
    tma_prefetch_desc(&tm_tok);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_units = *args.n_units;
  const uint64_t tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const int4 un = args.units[u];
        const bool two = un.z > 128;
        const int wr = un.x * args.w_rows_per_expert + un.w * 128;
        const uint32_t bytes = C::B_BYTES + (two ? 2 : 1) * C::HALF_A;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], bytes);
          const int kx = kb * KBlock<KIND>::ELEMS;
          tma_load_2d(sb, &tm_tok, &full[stage], kx, un.y, pol_x);
          if (two) tma_load_2d(sb + C::HALF_A, &tm_tok, &full[stage], kx, un.y + 128, pol_x);
          tma_load_2d(sb + C::A_BYTES, &tm_wg, &full[stage], kx, wr, pol_w);
          tma_load_2d(sb + C::A_BYTES + C::B_BYTES / 2, &tm_wu, &full[stage], kx, wr, pol_w);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load issued must land before the CTA exits
      const int pending = issued < C::STAGES ? issued : C::STAGES;
      for (int i = 0; i < pending; ++i) {
        if (stage == 0) {
          stage = C::STAGES - 1;
          phase ^= 1u;
        } else {
          --stage;
        }
        const volatile int never = 0;
        if (!mbar_wait_bounded(&full[stage], phase, tmo, &never)) gemm_fail(abort_flag);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f32acc<F8>(128, 256);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++it) {
        const bool two = args.units[u].z > 128;
        // the accumulator pair is free once the previous unit's epilogue read it
        if (!mbar_wait_bounded(tempty, (static_cast<uint32_t>(it) & 1u) ^ 1u, tmo, abort_flag)) {
          gemm_fail(abort_flag);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t da0 = sdesc_k128(sa);
          const uint64_t da1 = sdesc_k128(sa + C::HALF_A);
          const uint64_t db = sdesc_k128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            mma_ss<F8>(tmem_base, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            if (two) mma_ss<F8>(tmem_base + 256, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull);
      }
      mma_commit(mma_done);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quarter
    const int h = (warp - 2) >> 2;          // token half: accumulator columns [256 h, 256 h + 256)
    const int rloc = h * 128 + q * 32 + lane;
    int it = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
      const int4 un = args.units[u];
      bool ready = false;
      if (lane == 0) ready = mbar_wait_bounded(tfull, static_cast<uint32_t>(it) & 1u, tmo, abort_flag);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        if (lane == 0) gemm_fail(abort_flag);
        break;
      }
      tc_fence_after();
      if (h == 0 || un.z > 128) {
        const uint32_t tb = tmem_base + static_cast<uint32_t>(h * 256) +
                            (static_cast<uint32_t>(q * 32) << 16);
        const bool valid = rloc < un.z;
        const size_t row = static_cast<size_t>(un.y) + rloc;
        const float sx = (F8 && valid) ? args.row_scale[row] : 1.f;
        __nv_bfloat16* dst = args.out + row * args.out_ld + un.w * 128;
        const size_t wi0 = static_cast<size_t>(un.x) * args.w_rows_per_expert + un.w * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float g[32], v[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, v);
          if (F8) {
            // weight-row scales of these 32 columns (the same for every lane)
            const float4* sg4 = reinterpret_cast<const float4*>(args.w_scale0 + wi0 + c * 32);
            const float4* su4 = reinterpret_cast<const float4*>(args.w_scale1 + wi0 + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 a = __ldg(sg4 + j), b = __ldg(su4 + j);
              g[4 * j] *= a.x * sx; g[4 * j + 1] *= a.y * sx; g[4 * j + 2] *= a.z * sx; g[4 * j + 3] *= a.w * sx;
              v[4 * j] *= b.x * sx; v[4 * j + 1] *= b.y * sx; v[4 * j + 2] *= b.z * sx; v[4 * j + 3] *= b.w * sx;
            }
          }
          if (valid) {
            uint4 pk[4];
            __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a0 = __fdividef(g[2 * j], 1.0f + __expf(-g[2 * j])) * v[2 * j];
              const float a1 =
                  __fdividef(g[2 * j + 1], 1.0f + __expf(-g[2 * j + 1])) * v[2 * j + 1];
              p2[j] = __floats2bfloat162_rn(a0, a1);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = pk[j];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace beam
