// Wide 2-SM grouped expert GEMMs for many tokens per expert (prefill):
// tcgen05.mma.cta_group::2 on a two-CTA cluster, TWO weight tiles per CTA and
// one token tile shared by the pair.
//
// The layer's experts ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 专家混合模型): SwiGLU MLPs, hidden 5120, intermediate 2560, combined
// with the normalised router weights; the SwiGLU product in FP32 and the
// post-norm and residual in FP32 (section 残差流).
//
// A unit is (expert e, weight slice s, a group of n <= 256 tokens of e). The
// group's N = n rounded up to 16 tokens are the MMA's N operand: rows
// [0, N/2) in the even CTA, [N/2, N) in the odd one. Every K-step issues two
// pair MMAs (M = 256 each, 128 weight rows per CTA) into two TMEM
// accumulators that fill the 512 columns:
//   gate/up (MODE 0): slice s = intermediate rows i0 = 256 s; CTA r holds
//            W_g rows i0 + 128 r .. +127 (tile 0 -> D0) and W_u rows
//            i0 + 128 r .. +127 (tile 1 -> D1), so TMEM lane l of D0 and D1
//            hold g and u of the same row i and one thread computes
//            act[t, i] = bf16(silu(g) * u) (FP32 math).
//   down    (MODE 1): slice s = hidden rows h0 = 512 s; CTA r holds W_d rows
//            h0 + 128 r .. +127 (-> D0) and h0 + 256 + 128 r .. +127 (-> D1);
//            when H % 512 == 256 the last slice has only the first tile. The
//            epilogue adds w * y into the token's FP32 accumulator and
//            finalises completed tokens (kernels_combine.cuh).
// Per K-block a CTA loads 32 KB of weights and N/2 x 128 bytes of tokens and
// its tensor core computes a 128 x 2N block, so the shared-memory and L2
// traffic per FLOP is a quarter below that of one weight tile per CTA; the two
// accumulators alternate, so back-to-back MMAs never wait on each other.
// TMEM holds one unit's accumulators: the next unit's MMAs start once the
// epilogue has read them (it releases TMEM before its stores complete and
// before it finalises tokens).
//
// Roles per CTA (576 threads): warp 0 TMA producer; warp 1 TMEM allocation
// (both CTAs) and, in the even CTA, the MMA issuer; then sixteen epilogue
// warps, four per TMEM lane quarter (warp % 4), each taking every fourth
// 16-column chunk. Both CTAs' TMA loads count their bytes on the even CTA's
// `full` barrier; the MMA commits arrive on the `empty` and `tmem_full`
// barriers of both CTAs; all epilogue warps of both CTAs release TMEM on the
// even CTA's `tmem_empty` barrier. All
// waits are bounded; the CTAs meet at a cluster barrier before TMEM is freed
// and before exit.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_combine.cuh"
#include "kernels_gemm.cuh"
#include "ptx.cuh"

namespace beam {

struct WideArgs {
  const int4* units;        // {expert, first row, tokens n (1..256), weight slice}
  const int* n_units;
  int k_blocks;             // 128-byte K-blocks per unit (64 BF16 or 128 E4M3 elements)
  int w_rows_per_expert;    // I (gate/up) or H (down)
  __nv_bfloat16* act;       // MODE 0: [rows, act_ld]
  int act_ld;
  unsigned long long timeout_ns;
  // E4M3 operands: per token-row scale of x (MODE 0; in MODE 1 the activation
  // row scale is part of the combine coefficient) and per weight-row scales
  // (gate and up for MODE 0, down for MODE 1), indexed expert * rows + row
  const float* row_scale;
  const float* w_scale0;
  const float* w_scale1;
  CombineArgs comb;         // MODE 1
};

template <int EPI_WARPS_>
struct WideCfgT {
  static constexpr int STAGES = 4;
  static constexpr int A_BYTES = 128 * 128;      // one 128-row weight tile x 128 bytes
  static constexpr int B_BYTES = 128 * 128;      // up to 128 token rows x 128 bytes
  static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
  static constexpr int D1_COL = 256;             // second accumulator
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int NSUB = EPI_WARPS / 4;     // epilogue warps per lane quarter
  static constexpr int NCH = 16 / NSUB;          // 16-column chunks per warp and accumulator
  static constexpr int NG = NCH / 2;             // per-lane registers for 32 columns each
  static_assert(NSUB == 2 || NSUB == 4, "epilogue warps");
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int BAR_BYTES = (2 * STAGES + 3) * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};
// Four epilogue warps per lane quarter in both GEMMs: TMEM holds one unit,
// so the epilogue (SwiGLU and the act stores; the combine's reductions)
// stalls the next unit's MMAs, and more warps shorten it (E4M3 gate/up, whose
// units are half as long, 2.14 -> 1.97 ms at T = 8192; BF16 unchanged).
template <int MODE>
using WideCfg = WideCfgT<16>;

// Token rows of one CTA for a unit of N tokens: N/2 rows, a multiple of 8,
// loaded as 64-, 32-, 16- and 8-row boxes (the binary digits of N/2).
__device__ __forceinline__ void wide_load_tokens(uint8_t* dst, const CUtensorMap* t64,
                                                 const CUtensorMap* t32, const CUtensorMap* t16,
                                                 const CUtensorMap* t8, uint32_t bar, int kx,
                                                 int row0, int rows, uint64_t pol) {
  int r = 0;
  while (rows - r >= 64) {
    tma_load_2d_pair(dst + r * 128, t64, bar, kx, row0 + r, pol);
    r += 64;
  }
  if (rows - r >= 32) {
    tma_load_2d_pair(dst + r * 128, t32, bar, kx, row0 + r, pol);
    r += 32;
  }
  if (rows - r >= 16) {
    tma_load_2d_pair(dst + r * 128, t16, bar, kx, row0 + r, pol);
    r += 16;
  }
  if (rows - r >= 8) tma_load_2d_pair(dst + r * 128, t8, bar, kx, row0 + r, pol);
}

// F8: E4M3 operands (K-blocks of 128 elements, kind::f8f6f4) with the scales
// applied in the epilogue; else BF16 (K-blocks of 64).
template <int MODE, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(WideCfg<MODE>::THREADS, 1)
    expert_gemm_wide_kernel(const __grid_constant__ CUtensorMap tm_w0,
                            const __grid_constant__ CUtensorMap tm_w1,
                            const __grid_constant__ CUtensorMap tm_t64,
                            const __grid_constant__ CUtensorMap tm_t32,
                            const __grid_constant__ CUtensorMap tm_t16,
                            const __grid_constant__ CUtensorMap tm_t8, const WideArgs args) {
  using C = WideCfg<MODE>;
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
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * C::EPI_WARPS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_w0);
    if (MODE == 0) tma_prefetch_desc(&tm_w1);
    tma_prefetch_desc(&tm_t64);
    tma_prefetch_desc(&tm_t32);
    tma_prefetch_desc(&tm_t16);
    tma_prefetch_desc(&tm_t8);
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
      // weights at normal priority: an expert's second token group runs
      // the same weight slices in the adjacent units and re-reads them from
      // L2 (as evict-first lines they were often gone already)
      const uint64_t pol_w = l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = cid; ok && u < n_units; u += ncl) {
        const int4 un = args.units[u];
        const int rows = ((un.z + 15) & ~15) >> 1;   // this CTA's token rows (multiple of 8)
        const bool two = MODE == 0 || un.w * 512 + 512 <= args.w_rows_per_expert;
        const uint32_t cta_bytes = (two ? 2 : 1) * C::A_BYTES + rows * 128;
        const int tok0 = un.y + static_cast<int>(crank) * rows;
        const int base = un.x * args.w_rows_per_expert + static_cast<int>(crank) * 128;
        const int wr0 = (MODE == 0) ? base + un.w * 256 : base + un.w * 512;
        const int wr1 = (MODE == 0) ? wr0 : wr0 + 256;
        const CUtensorMap* m1 = (MODE == 0) ? &tm_w1 : &tm_w0;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE_BYTES;
          const uint32_t fbar = mapa_shared(&full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * cta_bytes);
          const int kx = kb * KBlock<F8>::ELEMS;
          tma_load_2d_pair(sb, &tm_w0, fbar, kx, wr0, pol_w);
          if (two) tma_load_2d_pair(sb + C::A_BYTES, m1, fbar, kx, wr1, pol_w);
          wide_load_tokens(sb + 2 * C::A_BYTES, &tm_t64, &tm_t32, &tm_t16, &tm_t8, fbar, kx, tok0,
                           rows, pol_x);
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
      const uint32_t d0 = tmem_base, d1 = tmem_base + C::D1_COL;
      for (int u = cid; ok && u < n_units; u += ncl, ++it) {
        const int4 un = args.units[u];
        const int N = (un.z + 15) & ~15;
        const bool two = MODE == 0 || un.w * 512 + 512 <= args.w_rows_per_expert;
        const uint32_t idesc = idesc_f32acc<F8>(256, N);
        // the previous unit's accumulators have been read by the epilogue
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
          const uint64_t da1 = sdesc_k128(sa + C::A_BYTES);
          const uint64_t db = sdesc_k128(sa + 2 * C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            mma_ss_pair<F8>(d0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            if (two) mma_ss_pair<F8>(d1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          mma_commit_pair_both(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(tfull);
      }
      mma_commit_pair_to(mma_done, 0);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp (q, sub) owns TMEM lane quarter q and the chunks of 16 columns
    // c = sub + NSUB * k, k = 0..NCH-1. Its local column l is column
    // (sub + NSUB * (l / 16)) * 16 + l % 16; lane j keeps the per-column
    // values of local columns j, j + 32, ..., fetched from global memory
    // before the accumulators are ready.
    const int q = warp & 3;                 // TMEM lane quarter
    const int sub = (warp - 2) >> 2;
    const int rloc = q * 32 + lane;         // TMEM lane = weight row of this CTA's tiles
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int it = 0;
    for (int u = cid; u < n_units; u += ncl, ++it) {
      const int4 un = args.units[u];
      const int n = un.z;
      const int nch = (n + 15) >> 4;
      // per-column values: MODE 0 the x row scale (E4M3), MODE 1 the token and
      // the combine coefficient
      int tkr[C::NG];
      float cfr[C::NG];
#pragma unroll
      for (int g = 0; g < C::NG; ++g) {
        const int l = g * 32 + lane;
        const int col = (sub + C::NSUB * (l >> 4)) * 16 + (l & 15);
        tkr[g] = -1;
        cfr[g] = 1.f;
        if (col < n) {
          const int r = un.y + col;
          if (MODE == 0) {
            if (F8) cfr[g] = args.row_scale[r];
          } else {
            tkr[g] = args.comb.row_token[r];
            cfr[g] = tkr[g] >= 0 ? combine_coef(args.comb, r) : 0.f;
          }
        }
      }
      bool ready = false;
      if (lane == 0) ready = mbar_wait_bounded(tfull, static_cast<uint32_t>(it) & 1u, tmo, abort_flag);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        if (lane == 0) gemm_fail(abort_flag);
        break;
      }
      tc_fence_after();
      if (MODE == 0) {
        const int i = un.w * 256 + static_cast<int>(crank) * 128 + rloc;
        float sg = 1.f, su = 1.f;
        if (F8) {
          const size_t wi = static_cast<size_t>(un.x) * args.w_rows_per_expert + i;
          sg = args.w_scale0[wi];
          su = args.w_scale1[wi];
        }
        // SwiGLU of this warp's chunks into registers (BF16 pairs; two local
        // chunks of both accumulators per TMEM wait), then TMEM is released
        // before the global stores, so the next unit's MMAs overlap them
        uint32_t ap[C::NCH][8];
#pragma unroll
        for (int k = 0; k < C::NCH; k += 2) {
          const int c0 = sub + C::NSUB * k;
          if (c0 < nch) {
            const int c1 = c0 + C::NSUB;
            float g0[16], u0[16], g1[16], u1[16];
            tmem_ld16x4(tq + c0 * 16, tq + C::D1_COL + c0 * 16, tq + c1 * 16,
                        tq + C::D1_COL + c1 * 16, g0, u0, g1, u1);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float* g = h2 ? g1 : g0;
              const float* v = h2 ? u1 : u0;
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                float a2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  float gj = g[j + e], uj = v[j + e];
                  if (F8) {
                    const float sx = __shfl_sync(0xffffffffu, cfr[(k + h2) >> 1],
                                                 (((k + h2) & 1) << 4) + j + e);
                    gj *= sg * sx;
                    uj *= su * sx;
                  }
                  a2[e] = __fdividef(gj, 1.0f + __expf(-gj)) * uj;
                }
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(a2[0], a2[1]);
                ap[k + h2][j >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty, 0));
        // act[t, i] for the chunks' tokens (a warp writes 64 contiguous bytes
        // of a token row per store)
#pragma unroll
        for (int k = 0; k < C::NCH; ++k) {
          const int c = sub + C::NSUB * k;
          if (c >= nch) break;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c * 16 + j;
            if (tok < n) {
              const uint32_t w2 = ap[k][j >> 1];
              const uint16_t h = static_cast<uint16_t>((j & 1) ? (w2 >> 16) : (w2 & 0xFFFFu));
              reinterpret_cast<uint16_t*>(args.act)[static_cast<size_t>(un.y + tok) * args.act_ld + i] = h;
            }
          }
        }
      } else {
        const CombineArgs& cb = args.comb;
        const int h0 = un.w * 512 + static_cast<int>(crank) * 128 + rloc;
        const int h1 = h0 + 256;
        const bool two = h1 < cb.H;   // the second tile exists (not a half slice)
        float s0 = 1.f, s1 = 1.f;
        if (F8) {
          const size_t wi = static_cast<size_t>(un.x) * args.w_rows_per_expert;
          s0 = args.w_scale0[wi + h0];
          if (two) s1 = args.w_scale0[wi + h1];
        }
#pragma unroll
        for (int k = 0; k < C::NCH; k += 2) {
          const int c0 = sub + C::NSUB * k;
          if (c0 >= nch) break;
          const int c1 = c0 + C::NSUB;
          float d0[16], e0[16], d1[16], e1[16];
          tmem_ld16x4(tq + c0 * 16, tq + C::D1_COL + c0 * 16, tq + c1 * 16,
                      tq + C::D1_COL + c1 * 16, d0, e0, d1, e1);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float* d = h2 ? d1 : d0;
            const float* e = h2 ? e1 : e0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int src = (((k + h2) & 1) << 4) + j;
              const int t = __shfl_sync(0xffffffffu, tkr[(k + h2) >> 1], src);
              const float w = __shfl_sync(0xffffffffu, cfr[(k + h2) >> 1], src);
              if (t >= 0) {
                float* o = cb.acc + static_cast<size_t>(t) * cb.H;
                red_add_f32(o + h0, w * (s0 * d[j]));
                if (two) red_add_f32(o + h1, w * (s1 * e[j]));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty, 0));
        // one arrival per token of this warp's columns (32 per register)
        combine_arrive_warp<C::NG>(cb, tkr);
      }
    }
    // finalise completed tokens (rows) once this warp's own units are done
    if (MODE == 1 && !combine_drain_warp(args.comb, lane, tmo, abort_flag) && lane == 0)
      gemm_fail(abort_flag);
  }

  tc_fence_before();
  cluster_sync_all();  // both CTAs done: no more loads, MMAs or arrivals into either
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace beam
