// Pair (2-SM) GEMM with per-row FP32 outputs: tcgen05.mma.cta_group::2 on a
// two-CTA cluster, the weights as the MMA's M = 256 operand (128 rows in each
// CTA) and up to 256 rows of the activation as N (N/2 rows in each CTA). It
// runs the router-logits GEMM of the tensor-core router (K-split, "Reflection
// 发布 Beam 501B 开源模型，支持 1M tokens 上下文", section 专家混合模型: an FP32
// router over all experts) and the attention sublayer's projections (section
// 注意力), each as one "expert" whose rows are the tokens.
//
// Each CTA holds only its half of both operands, so one K-block is 32 KB of
// shared memory per CTA (six stages fit). A unit is (expert or K-slice,
// weight tile m, a group of at most 256 rows); N is the group size rounded
// up to 32. Tile m = output columns h0 = 256m .. +255, CTA r holds weight
// rows h0+128r .. +127 and writes y[t, h] = D (FP32) as coalesced rows.
//
// Roles per CTA (192 threads): warp 0 TMA producer; warp 1 TMEM allocation
// (both CTAs) and, in the even CTA only, the MMA issuer; warps 2..5 epilogue.
// Both CTAs' TMA loads count their bytes on the even CTA's `full` barrier;
// the MMA commits arrive on the `empty` and `tmem_full` barriers of both
// CTAs; both CTAs' epilogues release an accumulator on the even CTA's
// `tmem_empty` barrier (count 8). All waits are bounded; the CTAs meet at a
// cluster barrier before TMEM is freed and before exit.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_gemm.cuh"
#include "ptx.cuh"

namespace beam {

struct PairArgs {
  const int4* units;        // {expert | K-split, first row, rows (<= 256), weight tile}
  const int* n_units;
  int k_blocks;             // 128-byte K-blocks per unit (64 BF16 or 128 E4M3 elements)
  int w_rows_per_expert;    // output columns per expert
  float* y;                 // [rows, out_ld]
  int out_ld;
  // K-split (router logits): unit.x is the split index ks; the unit covers
  // K-blocks [ks*k_blocks, (ks+1)*k_blocks) of A, B's K-block is the A
  // K-block modulo b_k_wrap (0: no wrap), and the output is y + ks*y_split.
  int k_split;              // 0: no split (unit.x is the expert)
  int b_k_wrap;
  size_t y_split;
  unsigned long long timeout_ns;
  // E4M3 operands only: per weight-row scales, indexed expert * w_rows_per_expert + row
  const float* w_scale0;
};

struct PairCfg {
  static constexpr int STAGES = 6;
  static constexpr int A_BYTES = 128 * 128;      // this CTA's 128 weight rows x 64
  static constexpr int B_BYTES = 128 * 128;      // up to 128 token rows x 64
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = 256;           // N <= 256
  static constexpr int NBUF = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int BAR_BYTES = (2 * STAGES + 2 * NBUF + 1) * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// F8: E4M3 operands (K-blocks of 128 elements, kind::f8f6f4) with the weight
// scales applied in the epilogue; else BF16 (K-blocks of 64).
template <bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a0,
                            const __grid_constant__ CUtensorMap tm_tok,
                            const __grid_constant__ CUtensorMap tm_tok64, const PairArgs args) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::NBUF;
  uint64_t* mma_done = tempty + C::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_a0);
    tma_prefetch_desc(&tm_tok);
    tma_prefetch_desc(&tm_tok64);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers and TMEM of both CTAs ready
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
      for (int u = cid; ok && u < n_units; u += ncl) {
        const int4 un = args.units[u];
        const int N = (un.z + 31) & ~31;
        const int rows = N >> 1;             // token rows of this CTA (multiple of 16)
        const int n64 = rows >> 6;           // 64-row boxes, then 16-row boxes
        const int n16 = (rows & 63) >> 4;
        const uint32_t cta_bytes = C::A_BYTES + rows * 128;
        const int tok0 = un.y + static_cast<int>(crank) * (N >> 1);
        const int expert = args.k_split ? 0 : un.x;
        const int kb0 = args.k_split ? un.x * args.k_blocks : 0;
        const int wrow = expert * args.w_rows_per_expert + un.w * 256 + static_cast<int>(crank) * 128;
        for (int kbl = 0; kbl < args.k_blocks; ++kbl) {
          const int kb = kb0 + kbl;
          const int kbb = args.b_k_wrap ? kb % args.b_k_wrap : kb;
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE_BYTES;
          const uint32_t fbar = mapa_shared(&full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * cta_bytes);
          const int kx = kb * KBlock<F8>::ELEMS, kbx = kbb * KBlock<F8>::ELEMS;
          tma_load_2d_pair(sb, &tm_a0, fbar, kx, wrow, pol_w);
          for (int j = 0; j < n64; ++j)
            tma_load_2d_pair(sb + C::A_BYTES + j * 8192, &tm_tok64, fbar, kbx, tok0 + j * 64,
                             pol_x);
          for (int j = 0; j < n16; ++j)
            tma_load_2d_pair(sb + C::A_BYTES + n64 * 8192 + j * 2048, &tm_tok, fbar, kbx,
                             tok0 + n64 * 64 + j * 16, pol_x);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The leader drains its full barriers (both CTAs' bytes land there);
      // the follower's loads complete on the leader's barriers, which the
      // leader's drain and the final cluster barrier cover.
      if (leader) {
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
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int u = cid; ok && u < n_units; u += ncl, ++it) {
        const int4 un = args.units[u];
        const int N = (un.z + 31) & ~31;
        const uint32_t idesc = idesc_f32acc<F8>(256, N);
        const int buf = it & 1;
        const uint32_t tpar = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], tpar ^ 1u, tmo, abort_flag)) {
          gemm_fail(abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t da = sdesc_k128(sa);
          const uint64_t db = sdesc_k128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_pair<F8>(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit_pair_both(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(&tfull[buf]);
      }
      mma_commit_pair_to(mma_done, 0);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter
    int it = 0;
    for (int u = cid; u < n_units; u += ncl, ++it) {
      const int4 un = args.units[u];
      const int buf = it & 1;
      const uint32_t tpar = static_cast<uint32_t>(it >> 1) & 1u;
      bool ready = false;
      if (lane == 0) ready = mbar_wait_bounded(&tfull[buf], tpar, tmo, abort_flag);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        if (lane == 0) gemm_fail(abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS) +
                          (static_cast<uint32_t>(q * 32) << 16);
      const int nch = (un.z + 15) >> 4;
      {
        const int h = un.w * 256 + static_cast<int>(crank) * 128 + q * 32 + lane;
        float* ybase = args.k_split ? args.y + static_cast<size_t>(un.x) * args.y_split : args.y;
        // E4M3: the weight-row scale
        const float sd = F8 ? args.w_scale0[static_cast<size_t>(un.x) * args.w_rows_per_expert + h] : 1.f;
        float* yrow = ybase + static_cast<size_t>(un.y) * args.out_ld + h;
        // 32 accumulator columns (tokens) per TMEM wait; the second half may
        // lie past N but stays inside this accumulator's 256 columns
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
          float d[16], e[16];
          tmem_ld16x2(tb + c * 16, tb + c * 16 + 16, d, e);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c * 16 + j;
            // the rows are read once, by the next step: stream them past L2
            if (tok < un.z) __stcs(yrow + static_cast<size_t>(tok) * args.out_ld, F8 ? d[j] * sd : d[j]);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c * 16 + 16 + j;
            if (tok < un.z) __stcs(yrow + static_cast<size_t>(tok) * args.out_ld, F8 ? e[j] * sd : e[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[buf], 0));
    }
  }

  tc_fence_before();
  cluster_sync_all();  // both CTAs done: no more loads, MMAs or arrivals into either
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace beam
