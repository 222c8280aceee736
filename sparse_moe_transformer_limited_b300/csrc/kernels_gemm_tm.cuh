// Token-major grouped expert GEMMs for many tokens per expert with NVFP4
// expert weights (prefill), on tcgen05 + TMEM.
//
// The layer's experts ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 专家混合模型): SwiGLU MLPs, hidden 5120, intermediate 2560, combined
// with the normalised router weights; the SwiGLU product in FP32 and the
// post-norm and residual in FP32 (section 残差流).
//
// A cluster unit is two sub-units, one per CTA of a two-CTA cluster, each
// (expert e, weight tile n, up to 128 consecutive rows of the expert-ordered
// token layout = the MMA's M). The weight tile has 256 rows (the MMA's N) and
// each CTA loads all of it into its own shared memory. In a PAIR unit both
// CTAs work on the same tile (rows [0,128) and [128,256) of a 256-row group),
// so the second read of the tile is served by L2 while the first is in
// flight; in a SOLO unit (an expert's last <= 128 rows) each CTA works on its
// own tile.
//   gate/up (MODE 0): tile n = intermediate rows [128n, 128n+128) of W_g
//            (half 0, TMEM columns 0..127) and of W_u (half 1, columns
//            128..255); epilogue act[row, 128n + i] = bf16(silu(g_i) * u_i)
//            with g_i and u_i read by the same thread (FP32 math).
//   down    (MODE 1): tile n = hidden rows [256n, 256n+256) of W_d; the
//            epilogue adds w * y into the token's FP32 accumulator and
//            finalises completed tokens (kernels_combine.cuh).
//
// NVFP4 (E2M1 codes with E4M3 scales per 16 elements, "NVFP4 版" section):
// a K-block is 256 elements (128 bytes per row); each stage also carries the
// K-block's scale groups -- four 512-byte groups of the 128-row token tile
// and eight of the two 128-row weight halves -- which the MMA thread copies
// into the stage's own TMEM columns (tcgen05.cp) before the block-scaled
// MMAs. TMEM then holds one accumulator (256 columns) and the scale columns
// of every stage (48 each), so the epilogue does not overlap the next unit.
// BF16 and E4M3 operands are also supported (K-blocks of 64 / 128 elements).
//
// Warp roles as in the weight-major kernel: warp 0 TMA producer, warp 1 TMEM
// owner and MMA issuer, warps 2..9 epilogue: two warps per TMEM lane quarter
// (warp % 4), one per half of the accumulator's columns. All waits are
// bounded; the CTAs of a cluster meet at a cluster barrier before TMEM is
// freed and before exit.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_combine.cuh"
#include "kernels_gemm.cuh"
#include "kernels_permute.cuh"
#include "ptx.cuh"

namespace beam {

struct TmArgs {
  const int4* units;        // 2 per cluster unit: {expert, first row, rows, tile | TM_PAIR}
  const int* n_units;
  int k_blocks;             // 128-byte K-blocks: K / 64 (BF16), K / 128 (E4M3), K / 256 (NVFP4)
  int w_rows_per_expert;    // I (gate/up) or H (down)
  __nv_bfloat16* out;       // MODE 0: act [R, I] bf16
  int out_ld;
  unsigned long long timeout_ns;
  // E4M3 operands only: per token-row scale (MODE 0; MODE 1 leaves the
  // activation row scale to the combine) and per weight-row scales (gate and
  // up for MODE 0, down for MODE 1), indexed expert * w_rows_per_expert + row
  const float* row_scale;
  const float* w_scale0;
  const float* w_scale1;
  // NVFP4: the same roles with one group scale per expert for the weights
  // (w_scale0/1 indexed by expert) and per token row (row_scale), plus the
  // 512-byte block-scale groups: token tiles of 128 rows (a_sf) and weight
  // tiles of 128 rows (w_sf0: gate or down, w_sf1: up), group (tile, K = 64
  // step) at byte (tile * K / 64 + step) * 512
  const uint8_t* a_sf;
  const uint8_t* w_sf0;
  const uint8_t* w_sf1;
  CombineArgs comb;         // MODE 1
};

template <int KIND>
struct TmCfg {
  static constexpr bool F4 = KIND == KIND_NVFP4;
  static constexpr int BM = 128;                 // token rows per CTA
  static constexpr int BN = 256;                 // weight rows per unit
  static constexpr int STAGES = 4;
  static constexpr int A_BYTES = BM * 128;       // 16 KB
  static constexpr int B_BYTES = BN * 128;       // 32 KB
  static constexpr int HALF_B = B_BYTES / 2;
  static constexpr int SF_A_BYTES = F4 ? 4 * 512 : 0;        // [K step][512]
  static constexpr int SF_B_BYTES = F4 ? 2 * 4 * 512 : 0;    // [weight half][K step][512]
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_A_BYTES + SF_B_BYTES;
  static constexpr int ACC_COLS = BN;
  static constexpr int NBUF = F4 ? 1 : 2;
  // per stage: A scales 4 columns per K step, B scales 8 (8-aligned)
  static constexpr int SF_COLS = F4 ? 48 : 0;
  static constexpr int SF_B_COL = 16;
  static constexpr int SF_TMEM_BASE = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(NBUF * ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "TMEM");
  static constexpr int BAR_BYTES = (2 * STAGES + 2 * NBUF + 1) * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// KIND_E4M3: E4M3 operands (K-blocks of 128 elements, kind::f8f6f4) with the
// scales applied in the epilogue; KIND_NVFP4: block-scaled E2M1 (K-blocks of
// 256, kind::mxf4nvf4) with the group scales in the epilogue; else BF16.
constexpr int TM_THREADS = 320;

template <int MODE, int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TM_THREADS, 1)
    expert_gemm_tm_kernel(const __grid_constant__ CUtensorMap tm_w0,
                          const __grid_constant__ CUtensorMap tm_w1,
                          const __grid_constant__ CUtensorMap tm_tok, const TmArgs args) {
  using C = TmCfg<KIND>;
  constexpr bool F8 = KIND == KIND_E4M3;
  constexpr bool F4 = KIND == KIND_NVFP4;
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
    tma_prefetch_desc(&tm_w0);
    if (MODE == 0) tma_prefetch_desc(&tm_w1);
    tma_prefetch_desc(&tm_tok);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers and TMEM ready in both CTAs
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
        const int4 un = args.units[2 * u + crank];
        const int nt = un.w & 0xFFFF;
        // weight rows of half 0 and half 1 of the 256-row tile
        const int wr0 = (MODE == 0) ? un.x * args.w_rows_per_expert + nt * 128
                                    : un.x * args.w_rows_per_expert + nt * 256;
        const int wr1 = (MODE == 0) ? wr0 : wr0 + 128;
        const CUtensorMap* wm1 = (MODE == 0) ? &tm_w1 : &tm_w0;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          // inner TMA coordinate in map elements: bf16 / e4m3 / bytes of e2m1 pairs
          const int kx = kb * (F4 ? 128 : KBlock<KIND>::ELEMS);
          tma_load_2d(sb, &tm_tok, &full[stage], kx, un.y, pol_x);
          tma_load_2d(sb + C::A_BYTES, &tm_w0, &full[stage], kx, wr0, pol_w);
          tma_load_2d(sb + C::A_BYTES + C::HALF_B, wm1, &full[stage], kx, wr1, pol_w);
          if (F4) {
            // this K-block's scale groups: token tile un.y / 128, weight tiles
            // of the two halves (each CTA loads all of them itself)
            const size_t ksteps = static_cast<size_t>(args.k_blocks) * 4;
            uint8_t* sf = sb + C::A_BYTES + C::B_BYTES;
            const uint8_t* srca = args.a_sf + ((static_cast<size_t>(un.y) >> 7) * ksteps + 4 * kb) * 512;
            const uint8_t* srcb0 = args.w_sf0 + ((static_cast<size_t>(wr0) >> 7) * ksteps + 4 * kb) * 512;
            const uint8_t* srcb1 = (MODE == 0 ? args.w_sf1 : args.w_sf0) +
                                   ((static_cast<size_t>(wr1) >> 7) * ksteps + 4 * kb) * 512;
            if (((reinterpret_cast<uintptr_t>(srca) | reinterpret_cast<uintptr_t>(srcb0) |
                  reinterpret_cast<uintptr_t>(srcb1)) & 15) != 0 || (un.y & 127) != 0) {
              // never issue a misaligned copy: flag it; the stage's wait then times out
              atomicOr(&g_beam_err, DEV_ERR_ALIGN);
            } else {
              bulk_load(sf, srca, 2048, &full[stage], pol_x);
              bulk_load(sf + C::SF_A_BYTES, srcb0, 2048, &full[stage], pol_w);
              bulk_load(sf + C::SF_A_BYTES + 2048, srcb1, 2048, &full[stage], pol_w);
            }
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
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
      const uint32_t idesc = F4 ? idesc_nvf4(128, C::BN) : idesc_f32acc<F8>(128, C::BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int u = cid; ok && u < n_units; u += ncl, ++it) {
        const int buf = (C::NBUF == 1) ? 0 : (it & 1);
        const uint32_t tpar = static_cast<uint32_t>((C::NBUF == 1) ? it : (it >> 1)) & 1u;
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
          if (F4) {
            // scales into this stage's TMEM columns, then the four K = 64 MMAs
            // (tcgen05 operations of one thread execute in issue order; a
            // stage's columns are rewritten only after its MMAs completed,
            // which the refill of the stage implies)
            const uint32_t slot = tmem_base + static_cast<uint32_t>(C::SF_TMEM_BASE + stage * C::SF_COLS);
            const uint32_t sf = sa + C::A_BYTES + C::B_BYTES;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tmem_cp_sf512(slot + 4 * kk, sdesc_sf512(sf + kk * 512));
              tmem_cp_sf512(slot + C::SF_B_COL + 8 * kk, sdesc_sf512(sf + C::SF_A_BYTES + kk * 512));
              tmem_cp_sf512(slot + C::SF_B_COL + 8 * kk + 4,
                            sdesc_sf512(sf + C::SF_A_BYTES + 2048 + kk * 512));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_nvf4_ss(d0, da + 2 * kk, db + 2 * kk, idesc, slot + 4 * kk,
                          slot + C::SF_B_COL + 8 * kk, (kb | kk) != 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss<F8>(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[buf]);
      }
      mma_commit(mma_done);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;   // accumulator columns of this warp
    const int rloc = q * 32 + lane;
    int it = 0;
    for (int u = cid; u < n_units; u += ncl, ++it) {
      const int4 un = args.units[2 * u + crank];
      const int nt = un.w & 0xFFFF;
      const int buf = (C::NBUF == 1) ? 0 : (it & 1);
      const uint32_t tpar = static_cast<uint32_t>((C::NBUF == 1) ? it : (it >> 1)) & 1u;
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
      const bool valid = rloc < un.z;
      const size_t row = static_cast<size_t>(un.y) + rloc;
      const float sx = ((F8 || F4) && MODE == 0 && valid) ? args.row_scale[row] : 1.f;
      // NVFP4: one group scale per expert and weight matrix
      const float es0 = F4 ? args.w_scale0[un.x] : 1.f;
      const float es1 = (F4 && MODE == 0) ? args.w_scale1[un.x] : 1.f;
      // The warp's whole accumulator slice (128 columns) into registers, then
      // the accumulator is released at once: the next unit's MMAs overlap the
      // math and the stores below.
      float acc[128];
      if (MODE == 0) {
        float* g = acc;
        float* v = acc + 64;
        tmem_ld64(tb + 64 * half, *reinterpret_cast<float(*)[64]>(g));
        tmem_ld64(tb + 128 + 64 * half, *reinterpret_cast<float(*)[64]>(v));
      } else {
        tmem_ld128(tb + 128 * half, acc);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (MODE == 0) {
        // gate columns 64 half + [0, 64) in acc[0..63], up in acc[64..127]
        __nv_bfloat16* dst = args.out + row * args.out_ld + nt * 128 + 64 * half;
        const size_t wi0 = static_cast<size_t>(un.x) * args.w_rows_per_expert + nt * 128 + 64 * half;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* g = acc + c * 16;
          float* v = acc + 64 + c * 16;
          if (F8) {
            // weight-row scales of these 16 columns (the same for every lane)
            const float4* sg4 = reinterpret_cast<const float4*>(args.w_scale0 + wi0 + c * 16);
            const float4* su4 = reinterpret_cast<const float4*>(args.w_scale1 + wi0 + c * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 a = __ldg(sg4 + j), b = __ldg(su4 + j);
              g[4 * j] *= a.x * sx; g[4 * j + 1] *= a.y * sx; g[4 * j + 2] *= a.z * sx; g[4 * j + 3] *= a.w * sx;
              v[4 * j] *= b.x * sx; v[4 * j + 1] *= b.y * sx; v[4 * j + 2] *= b.z * sx; v[4 * j + 3] *= b.w * sx;
            }
          }
          if (F4) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g[j] *= es0 * sx;
              v[j] *= es1 * sx;
            }
          }
          if (valid) {
            uint4 pk[2];
            __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float a0 = __fdividef(g[2 * j], 1.0f + __expf(-g[2 * j])) * v[2 * j];
              const float a1 =
                  __fdividef(g[2 * j + 1], 1.0f + __expf(-g[2 * j + 1])) * v[2 * j + 1];
              p2[j] = __floats2bfloat162_rn(a0, a1);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 16);
            d4[0] = pk[0];
            d4[1] = pk[1];
          }
        }
      } else {
        // fused combine: this thread's token row, 128 hidden columns
        const CombineArgs& cb = args.comb;
        const int tk = valid ? cb.row_token[row] : -1;
        const float cf = tk >= 0 ? combine_coef(cb, static_cast<int>(row)) : 0.f;
        float* dst = tk >= 0 ? cb.acc + static_cast<size_t>(tk) * cb.H + nt * 256 + 128 * half : nullptr;
        const size_t wi0 = static_cast<size_t>(un.x) * args.w_rows_per_expert + nt * 256 + 128 * half;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float* d = acc + c * 16;
          if (F8) {
            const float4* sd4 = reinterpret_cast<const float4*>(args.w_scale0 + wi0 + c * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 a = __ldg(sd4 + j);
              d[4 * j] *= a.x; d[4 * j + 1] *= a.y; d[4 * j + 2] *= a.z; d[4 * j + 3] *= a.w;
            }
          }
          if (F4) {
#pragma unroll
            for (int j = 0; j < 16; ++j) d[j] *= es0;
          }
          if (tk >= 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              red_add_v4_f32(dst + c * 16 + 4 * j, cf * d[4 * j], cf * d[4 * j + 1], cf * d[4 * j + 2],
                             cf * d[4 * j + 3]);
          }
        }
        combine_arrive_warp(cb, tk, lane);
      }
    }
    // finalise completed tokens (rows) once this warp's own units are done
    if (MODE == 1 && !combine_drain_warp(args.comb, lane, tmo, abort_flag) && lane == 0)
      gemm_fail(abort_flag);
  }

  tc_fence_before();
  cluster_sync_all();  // both CTAs done before TMEM is freed
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace beam
