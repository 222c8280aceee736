// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA.
//
// Each expert of the layer is a SwiGLU MLP with hidden 5120 and intermediate
// 2560 ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文", section
// 专家混合模型); its outputs are combined with the normalised router weights.
// The SwiGLU product runs in FP32 (same page, section 残差流).
//
// Both GEMMs put the WEIGHTS in the MMA's M=128 operand and the tokens of one
// expert in the N operand (16..NT columns), so one instruction shape serves
// decode (2-3 tokens per expert) and prefill (hundreds):
//   gate/up  (MODE 0): unit = (expert e, 128 intermediate rows m, token tile)
//            D_g[i,t] = sum_h Wg[e, m*128+i, h] * Xp[t, h]  (TMEM cols [0,NT))
//            D_u[i,t] = sum_h Wu[e, m*128+i, h] * Xp[t, h]  (TMEM cols [NT,2NT))
//            epilogue: act[t, m*128+i] = bf16(silu(D_g) * D_u)   (FP32 math)
//   down     (MODE 1): unit = (expert e, 128 hidden rows m, token tile)
//            D[h,t] = sum_i Wd[e, m*128+h, i] * act[t, i]
//            (NVFP4 with small token tiles: 256 hidden rows m*256.. as two
//            128-row tiles into two accumulators, like gate/up: the block
//            scales' TMEM copies and the MMAs of a K-block then move twice
//            the weight bytes, and the two accumulators alternate)
//            epilogue: o[token(t), m*128+h] += w_t * D[h,t] (FP32), the
//            router-weighted combine, then the post-norm and residual of
//            every completed token (kernels_combine.cuh)
//
// Warp roles (192 threads, persistent, one CTA per SM):
//   warp 0      TMA producer (one elected lane): fills a STAGES-deep smem ring
//   warp 1      TMEM owner and MMA issuer (one elected lane)
//   warps 2..5  epilogue: tcgen05.ld from TMEM lane quarter (warp % 4)
// The accumulator is double-buffered in TMEM when it fits, so the epilogue of
// one unit overlaps the main loop of the next.
//
// Every wait is bounded (global timer); on expiry the waiter raises a shared
// abort flag and the device error word, every role drains and the CTA exits
// normally after its in-flight TMA loads have landed.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_combine.cuh"
#include "ptx.cuh"

namespace beam {

__device__ int g_beam_err;  // per-device error word, read by beam_status()
constexpr int DEV_ERR_TIMEOUT = 1;
constexpr int DEV_ERR_ALIGN = 2;  // a bulk copy address was not 16-byte aligned (copy skipped)

struct GemmArgs {
  const int4* units;          // token tiles {expert, first row, rows, 0} (MODE 0/1)
  const int* n_units;         // device count of units
  int k_blocks;               // K / 64 (BF16) or K / 128 (E4M3): 128-byte K-blocks
  int a_rows_per_expert;      // I (gate/up) or H (down)
  __nv_bfloat16* out;         // MODE 0: act [R, I] bf16
  int out_ld;
  int m_tiles;                // weight row-tiles per token tile (I/128 or H/128)
  unsigned long long timeout_ns;
  // E4M3 and NVFP4 operands: FP32 scale of each token row of x (MODE 0; in
  // MODE 1 the activation row scale is a factor of the whole output row,
  // applied by the combine), and the weight scales (gate and up for MODE 0,
  // down for MODE 1): E4M3 one per weight row, indexed expert *
  // a_rows_per_expert + row; NVFP4 one per expert matrix, indexed by expert.
  const float* row_scale;
  const float* w_scale0;
  const float* w_scale1;
  // NVFP4 only: 512-byte block-scale groups (one K = 64 step of a row tile),
  // [rows / tile][K / 64][512], of the weights (gate / up or down; tile 128)
  // and of the expert-ordered token rows (tile NT)
  const uint8_t* a_sf0;
  const uint8_t* a_sf1;
  const uint8_t* b_sf;
  CombineArgs comb;           // MODE 1
};

// Weight rows of one unit: 128, or 256 for the NVFP4 down GEMM on token
// tiles of at most 64 (two weight tiles per unit, see above).
template <int MODE, int NT, int KIND>
struct UnitRows {
  static constexpr int value = (MODE == 1 && KIND == KIND_NVFP4 && NT <= 64) ? 256 : 128;
};

// Unit u of a GEMM: token tile u / m_tiles of the tile list and weight
// row-tile u % m_tiles.
template <int MODE, int NT>
__device__ __forceinline__ int4 gemm_unit(const GemmArgs& a, int u) {
  const int m = u % a.m_tiles, j = u / a.m_tiles;
  const int4 t = a.units[j];
  return make_int4(t.x, t.y, t.z, m);
}

// Unit u, or an empty unit past the end of the list.
template <int MODE, int NT>
__device__ __forceinline__ int4 gemm_unit_or_none(const GemmArgs& a, int u, int n_units) {
  return u < n_units ? gemm_unit<MODE, NT>(a, u) : make_int4(0, 0, 0, 0);
}

__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int MODE, int NT, int STAGES, int KIND = KIND_BF16>
struct GemmCfg {
  static_assert(MODE == 0 || MODE == 1, "mode");
  // two weight tiles per K-block: gate and up, or two down tiles (UnitRows)
  static constexpr bool TWO_A = MODE == 0 || UnitRows<MODE, NT, KIND>::value == 256;
  static constexpr int A_TILE = 128 * 128;  // 128 rows x 128 bytes (64 bf16, 128 e4m3, 256 e2m1)
  static constexpr int A_BYTES = (TWO_A ? 2 : 1) * A_TILE;
  static constexpr int B_BYTES = NT * 128;  // NT rows x 128 bytes
  // NVFP4: per stage the block scales of the K-block (four 512-byte groups
  // per operand matrix) follow the operand tiles
  static constexpr int SF_A_BYTES = KIND == KIND_NVFP4 ? (TWO_A ? 2 : 1) * 2048 : 0;
  static constexpr int SF_B_BYTES = KIND == KIND_NVFP4 ? 2048 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_A_BYTES + SF_B_BYTES;
  static constexpr int ACC_COLS = (TWO_A ? 2 : 1) * NT;
  // NVFP4: each stage has its own TMEM columns for the scales it copies in
  // (four columns per group), after the accumulators
  static constexpr int SF_COLS = KIND == KIND_NVFP4 ? 4 * 4 * (TWO_A ? 3 : 2) : 0;
  static constexpr int SF_B_COL = KIND == KIND_NVFP4 ? 16 * (TWO_A ? 2 : 1) : 0;
  static constexpr int NBUF = (2 * ACC_COLS + STAGES * SF_COLS <= 512) ? 2 : 1;
  static constexpr int SF_TMEM_BASE = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS =
      KIND == KIND_NVFP4 ? 512 : pow2_at_least(NBUF * ACC_COLS);
  static constexpr int BAR_BYTES = (2 * STAGES + 2 * NBUF + 1) * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "token tile");
  static_assert(NBUF * ACC_COLS + STAGES * SF_COLS <= 512 && TMEM_COLS <= 512, "TMEM");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void gemm_fail(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_beam_err, DEV_ERR_TIMEOUT);
}

// KIND_E4M3: both operands E4M3 (K-blocks of 128 elements, kind::f8f6f4);
// KIND_NVFP4: both packed E2M1 (K-blocks of 256 elements) with E4M3 scales
// per 16 elements copied from shared memory into TMEM by the MMA thread
// (kind::mxf4nvf4 block_scale); the epilogue applies the row and weight
// scales. KIND_BF16: K-blocks of 64.
template <int MODE, int NT, int STAGES, int KIND>
__global__ void __launch_bounds__(192, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                       const __grid_constant__ CUtensorMap tm_a1,
                       const __grid_constant__ CUtensorMap tm_b, const GemmArgs args) {
  using C = GemmCfg<MODE, NT, STAGES, KIND>;
  constexpr bool F8 = KIND == KIND_E4M3;
  constexpr bool F4 = KIND == KIND_NVFP4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + C::NBUF;
  uint64_t* mma_done = tempty + C::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_a0);
    if (MODE == 0) tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b);
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
      // each unit's descriptor is fetched one unit ahead (here and in the
      // other roles), so its global load overlaps the previous unit's work
      int4 un_next = gemm_unit_or_none<MODE, NT>(args, blockIdx.x, n_units);
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const int4 un = un_next;
        un_next = gemm_unit_or_none<MODE, NT>(args, u + gridDim.x, n_units);
        const int nb16 = (un.z + 15) >> 4;
        const uint32_t bytes = C::A_BYTES + nb16 * 2048 + C::SF_A_BYTES + C::SF_B_BYTES;
        const int arow = un.x * args.a_rows_per_expert + un.w * UnitRows<MODE, NT, KIND>::value;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], bytes);
          // inner TMA coordinate in elements of the map: bf16 / e4m3 / bytes of e2m1 pairs
          const int kx = kb * (F4 ? 128 : KBlock<KIND>::ELEMS);
          tma_load_2d(sb, &tm_a0, &full[stage], kx, arow, pol_w);
          if (MODE == 0) tma_load_2d(sb + C::A_TILE, &tm_a1, &full[stage], kx, arow, pol_w);
          else if (C::TWO_A) tma_load_2d(sb + C::A_TILE, &tm_a0, &full[stage], kx, arow + 128, pol_w);
          for (int j = 0; j < nb16; ++j)
            tma_load_2d(sb + C::A_BYTES + j * 2048, &tm_b, &full[stage], kx, un.y + j * 16,
                        pol_x);
          if (F4) {
            // the K-block's four scale groups of the weight tile and of the
            // 128-row token tile holding this unit's rows
            const size_t ksteps = static_cast<size_t>(args.k_blocks) * 4;
            const size_t a_off = ((static_cast<size_t>(arow) >> 7) * ksteps + 4 * kb) * 512;
            const size_t b_off = (static_cast<size_t>(un.y / NT) * ksteps + 4 * kb) * 512;
            uint8_t* sf = sb + C::A_BYTES + C::B_BYTES;
            const uint8_t* src0 = args.a_sf0 + a_off;
            // the second tile: gate/up -> up's scales; down -> the next 128-row tile's
            const uint8_t* src1 = MODE == 0 ? args.a_sf1 + a_off : src0 + (C::TWO_A ? ksteps * 512 : 0);
            const uint8_t* srcb = args.b_sf + b_off;
            if (((reinterpret_cast<uintptr_t>(src0) | reinterpret_cast<uintptr_t>(src1) |
                  reinterpret_cast<uintptr_t>(srcb)) & 15) != 0) {
              // never issue a misaligned bulk copy: flag it; the stage's wait then times out
              atomicOr(&g_beam_err, DEV_ERR_ALIGN);
            } else {
              bulk_load(sf, src0, 2048, &full[stage], pol_w);
              if (C::TWO_A) bulk_load(sf + 2048, src1, 2048, &full[stage], pol_w);
              bulk_load(sf + C::SF_A_BYTES, srcb, 2048, &full[stage], pol_x);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every load issued must have landed before the CTA may exit.
      const int pending = issued < STAGES ? issued : STAGES;
      for (int i = 0; i < pending; ++i) {
        if (stage == 0) {
          stage = STAGES - 1;
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
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      int4 un_next = gemm_unit_or_none<MODE, NT>(args, blockIdx.x, n_units);
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++it) {
        const int4 un = un_next;
        un_next = gemm_unit_or_none<MODE, NT>(args, u + gridDim.x, n_units);
        const int buf = (C::NBUF == 1) ? 0 : (it & 1);
        const uint32_t tpar = static_cast<uint32_t>((C::NBUF == 1) ? it : (it >> 1)) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], tpar ^ 1u, tmo, abort_flag)) {
          gemm_fail(abort_flag);
          break;
        }
        tc_fence_after();
        // N: the unit's tokens rounded up to 16 (NVFP4: to 32; the token
        // tile's scale groups start at column 0 of the unit's TMEM slot)
        const int n16 = F4 ? ((un.z + 31) & ~31) : ((un.z + 15) & ~15);
        const uint32_t idesc = F4 ? idesc_nvf4(128, n16) : idesc_f32acc<F8>(128, n16);
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t da0 = sdesc_k128(sa);
          const uint64_t da1 = sdesc_k128(sa + C::A_TILE);
          const uint64_t db = sdesc_k128(sa + C::A_BYTES);
          if (F4) {
            // scales into this stage's TMEM columns, then the four K = 64 MMAs
            // (tcgen05 operations of one thread execute in issue order)
            const uint32_t slot = tmem_base + static_cast<uint32_t>(C::SF_TMEM_BASE + stage * C::SF_COLS);
            const uint32_t sf = sa + C::A_BYTES + C::B_BYTES;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tmem_cp_sf512(slot + 4 * kk, sdesc_sf512(sf + kk * 512));
              if (C::TWO_A) tmem_cp_sf512(slot + 16 + 4 * kk, sdesc_sf512(sf + 2048 + kk * 512));
              tmem_cp_sf512(slot + C::SF_B_COL + 4 * kk, sdesc_sf512(sf + C::SF_A_BYTES + kk * 512));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
              const uint32_t sfb = slot + C::SF_B_COL + 4 * kk;
              mma_nvf4_ss(d0, da0 + 2 * kk, db + 2 * kk, idesc, slot + 4 * kk, sfb, accum);
              if (C::TWO_A)
                mma_nvf4_ss(d0 + NT, da1 + 2 * kk, db + 2 * kk, idesc, slot + 16 + 4 * kk, sfb, accum);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
              mma_ss<F8>(d0, da0 + 2 * kk, db + 2 * kk, idesc, accum);
              if (C::TWO_A) mma_ss<F8>(d0 + NT, da1 + 2 * kk, db + 2 * kk, idesc, accum);
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[buf]);
      }
      // Every MMA issued by this thread must complete before TMEM is freed.
      mma_commit(mma_done);
      const volatile int never = 0;
      if (!mbar_wait_bounded(mma_done, 0, tmo, &never)) gemm_fail(abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int rloc = q * 32 + lane;
    int it = 0;
    int4 un_next = gemm_unit_or_none<MODE, NT>(args, blockIdx.x, n_units);
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
      const int4 un = un_next;
      un_next = gemm_unit_or_none<MODE, NT>(args, u + gridDim.x, n_units);
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
      const int nch = (un.z + 15) >> 4;
      const int col = un.w * UnitRows<MODE, NT, KIND>::value + rloc;
      float ws0 = 1.f, ws1 = 1.f;
      if (F8 || F4) {
        const size_t wi = F8 ? static_cast<size_t>(un.x) * args.a_rows_per_expert + col
                             : static_cast<size_t>(un.x);
        ws0 = args.w_scale0[wi];
        if (MODE == 0) ws1 = args.w_scale1[wi];
      }
      for (int c = 0; c < nch; ++c) {
        if (MODE == 0) {
          float g[16], v[16];
          tmem_ld16x2(tb + c * 16, tb + NT + c * 16, g, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = c * 16 + j;
            if (tok < un.z) {
              float gj = g[j], uj = v[j];
              if (F8 || F4) {
                const float sx = args.row_scale[un.y + tok];
                gj *= ws0 * sx;
                uj *= ws1 * sx;
              }
              const float a = gj / (1.0f + expf(-gj)) * uj;
              args.out[static_cast<size_t>(un.y + tok) * args.out_ld + col] =
                  __float2bfloat16_rn(a);
            }
          }
        } else {
          // fused combine: o[token, col] += w * D (lanes 0..15 fetch the
          // token and coefficient of the chunk's columns)
          const CombineArgs& cb = args.comb;
          float d[16], d2[16];
          if (C::TWO_A)
            tmem_ld16x2(tb + c * 16, tb + NT + c * 16, d, d2);   // rows col and col + 128
          else
            tmem_ld16(tb + c * 16, d);
          int tk = -1;
          float cf = 0.f;
          if (lane < 16 && c * 16 + lane < un.z) {
            const int r = un.y + c * 16 + lane;
            tk = cb.row_token[r];
            if (tk >= 0) cf = combine_coef(cb, r);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = __shfl_sync(0xffffffffu, tk, j);
            const float w = __shfl_sync(0xffffffffu, cf, j);
            if (t >= 0) {
              float* o = args.comb.acc + static_cast<size_t>(t) * cb.H + col;
              red_add_f32(o, w * (ws0 * d[j]));
              if (C::TWO_A) red_add_f32(o + 128, w * (ws0 * d2[j]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (MODE == 1 && !args.comb.grid_done) {
        // one arrival per token of the unit (32 columns per call)
#pragma unroll 1
        for (int c = 0; c < un.z; c += 32) {
          const int col_t = c + lane;
          const int tk = col_t < un.z ? args.comb.row_token[un.y + col_t] : -1;
          combine_arrive_warp(args.comb, tk, lane);
        }
      }
    }
    // finalise completed tokens (rows) once this warp's own units are done
    if (MODE == 1) {
      const bool fin = args.comb.grid_done
                           ? combine_grid_finish(args.comb, lane, static_cast<int>(blockIdx.x) * 4 + (warp - 2),
                                                 static_cast<int>(gridDim.x) * 4, tmo, abort_flag)
                           : combine_drain_warp(args.comb, lane, tmo, abort_flag);
      if (!fin && lane == 0) gemm_fail(abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// A kernel that waits on a barrier nothing completes, with the bounded wait
// above; used to test the timeout path without hanging the GPU.
__global__ void debug_wait_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, timeout_ns, &abort_flag)) atomicOr(&g_beam_err, DEV_ERR_TIMEOUT);
  }
}

}  // namespace beam
