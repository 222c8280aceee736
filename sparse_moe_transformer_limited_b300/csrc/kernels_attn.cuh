// Attention sublayer ("Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
// section 注意力: grouped-query attention with 48 query and 8 key/value heads,
// RMSNorm on queries and keys, a sliding window of 512 tokens on most layers
// with RoPE, full context on every sixth layer and the last with the query
// scale (1 + (pos + 1) / 2048) ** 0.1 instead of positions, and a sigmoid
// gate from the layer input on every head channel before the output
// projection; section 残差流: RoPE and the query scaling in FP32). Head
// dimension 128 ("config.json" of the release, head_dim).
//
//   attn_prep_kernel       QK-RMSNorm, RoPE or query scale, from the FP32
//                          fused projection
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
// (value slots are written by attn_vt_kernel; the gate's sigmoid is taken
// by flash_attn_kernel's epilogue straight from the projection)
// window > 0: RoPE (theta) on q and k; window == 0: q *= (1 + (t+1)/2048)^0.1.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) attn_prep_kernel(
    const float* __restrict__ proj, int T, int Tp, int nq, int nkv,
    const float* __restrict__ q_gain, const float* __restrict__ k_gain, float eps, int window,
    const float2* __restrict__ rope_cs, __nv_bfloat16* __restrict__ q,
    __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ vt) {
  const int t = blockIdx.x;
  const int slot = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nslots = 2 * nq + 2 * nkv;
  if (t >= T || slot >= nslots) return;
  const float* src = proj + static_cast<size_t>(t) * nslots * ATT_D + static_cast<size_t>(slot) * ATT_D;
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = src[lane + 32 * i];
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
    // rotate-half RoPE: pairs (c, c + 64) for c = lane and lane + 32, the
    // (cos, sin) of token t and pair c from rope_table_kernel
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = lane + 32 * i;
      const float2 r = rope_cs[static_cast<size_t>(t) * (ATT_D / 2) + c];
      const float x1 = v[i], x2 = v[i + 2];
      v[i] = x1 * r.x - x2 * r.y;
      v[i + 2] = x2 * r.x + x1 * r.y;
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

// RoPE (cos, sin) of every token t and channel pair c (0..63): angle
// t * theta^(-2c/128) in FP32, shared by all query and key heads.
__global__ void rope_table_kernel(int T, float rope_theta, float2* __restrict__ cs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * (ATT_D / 2)) return;
  const int t = i / (ATT_D / 2), c = i % (ATT_D / 2);
  const float inv_freq = powf(rope_theta, -2.0f * static_cast<float>(c) / static_cast<float>(ATT_D));
  float sn, co;
  sincosf(static_cast<float>(t) * inv_freq, &sn, &co);
  cs[i] = make_float2(co, sn);
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
// Flash attention on tcgen05, persistent: one CTA per SM walks a static
// share of the (query tile of 128 rows, query head) work items, heaviest
// first (a causal layer's last query tiles see the most keys). Tiles are
// numbered across the CTA's items, so every ring, buffer and barrier below
// runs on without a break from one item to the next: the next item's Q is
// loaded and its first S computed while the previous item's last tiles and
// output are still in progress.
// Warp 0: TMA producer of Q (two buffers, one per item parity) and of K
// tiles of 128 keys into a two-stage ring (a stage is freed as soon as its S
// has been computed); the last warp: TMA producer of V^T tiles into a
// two-stage ring (freed after P V). Warp 1: TMEM owner and MMA issuer: per
// item S_0 and S_1 into two of three TMEM S buffers; then per tile j, as
// soon as P_j is written: O += P_j V_j (P_j read from TMEM as the MMA's A
// operand) with its K steps alternating with those of S_{j+2}, whose buffer
// held the previous tile's P (one thread's MMAs execute in issue order, so
// S_{j+2} overwrites it only after its P V has read it). The two
// accumulators (O and an S buffer) take turns, so no MMA waits on the one
// before it into the same TMEM, and S_{j+1} is ready while tile j+1's
// softmax runs. An item's first P V (which overwrites O) waits until the
// softmax warps have read the previous item's O. Warps 2..: ATT_PARTS warps
// per 32-row TMEM lane quarter, each for ATT_KW consecutive keys of the tile
// (and the matching columns of O); thread = (query row, part). Per tile: read
// the part of the S row, mask (boundary tiles only), row maximum over all
// parts (exchanged through shared memory), online softmax in base 2 with a
// lazy reference: m moves (and the O row is rescaled) only when a tile's
// maximum exceeds it by more than ATT_TAU2, so P <= 2^TAU2; P goes as BF16
// pairs over the first 64 columns of its own S buffer (every warp of a lane
// quarter has read its part of S before any writes P). At the end of an
// item O / l times the gate, BF16, to `out`.
// TMEM columns: S/P buffers [0,128), [128,256), [256,384); O [384,512).
// All waits are bounded; on expiry the error word is set and every role
// leaves after its in-flight copies and MMAs have completed. The two warps of
// a lane quarter meet at named barriers the same number of times whatever
// happens (no early exit from the tile loop), so those barriers cannot hang.
// ---------------------------------------------------------------------------
constexpr float ATT_TAU2 = 8.0f;        // lazy-rescale threshold, base-2 units
constexpr int ATT_SBUF = 3;             // S / P buffers in TMEM
constexpr uint32_t ATT_O_COL = ATT_SBUF * 128;
constexpr float ATT_LOG2E = 1.4426950408889634f;
constexpr int ATT_PARTS = 2;                      // softmax warps per TMEM lane quarter
constexpr int ATT_KW = ATT_BK / ATT_PARTS;        // keys (and O columns) per softmax warp
constexpr int ATT_SOFTMAX_WARPS = 4 * ATT_PARTS;
static_assert(ATT_KW == 32 || ATT_KW == 64, "softmax split");
constexpr int ATT_VWARP = 2 + ATT_SOFTMAX_WARPS;   // the V^T producer warp (the last)
constexpr int ATT_THREADS = 32 * (3 + ATT_SOFTMAX_WARPS);

struct AttnArgs {
  int T, Tp, nq, nkv, window;
  int n_qt;                    // query tiles per head (Tp / 128)
  int n_items;                 // n_qt * nq work items
  float scale;                 // 1 / sqrt(head_dim)
  const float* gate;           // gate logits: row t at gate + t * gate_ld, head h at + h * 128
  int gate_ld;                 // floats per row of the fused projection
  __nv_bfloat16* out;          // [T][nq * 128]
  unsigned long long timeout_ns;
};

struct AttnCfg {
  static constexpr int Q_BYTES = ATT_BQ * ATT_D * 2;     // 32 KB: two 64-channel blocks
  static constexpr int K_BYTES = ATT_BK * ATT_D * 2;     // 32 KB
  static constexpr int V_BYTES = ATT_D * ATT_BK * 2;     // 32 KB (V^T: 128 channels x 128 keys)
  // two Q buffers (the next item's Q loads while this one's S MMAs run);
  // K: S_{t+2} reads stage t % 2 once S_t has released it
  static constexpr int Q_STAGES = 2, K_STAGES = 2, V_STAGES = 2;
  static_assert(K_STAGES <= 3 && Q_STAGES <= 2, "barrier slots");
  // row maxima: [tile parity][part][row]; row sums: [part][row]
  static constexpr int XCH_BYTES = 3 * ATT_PARTS * ATT_BQ * 4;
  static constexpr int BAR_BYTES = 32 * 8;
  static constexpr int SMEM_BYTES = 1024 + Q_STAGES * Q_BYTES + K_STAGES * K_BYTES +
                                    V_STAGES * V_BYTES + XCH_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Work item it: query tile and head, the heaviest query tiles first.
__device__ __forceinline__ void attn_item(const AttnArgs& a, int it, int* qt, int* h) {
  *qt = a.n_qt - 1 - it / a.nq;
  *h = it % a.nq;
}

// First and one-past-last key tile of query tile qt.
__device__ __forceinline__ void attn_key_tiles(int qt, int T, int window, int* j0, int* j1) {
  const int q0 = qt * ATT_BQ;
  const int qlast = min(q0 + ATT_BQ, T) - 1;
  const int kfirst = window > 0 ? max(0, q0 - window + 1) : 0;
  *j0 = kfirst / ATT_BK;
  *j1 = qlast / ATT_BK + 1;
}

// Packed FP32 pair arithmetic (two lanes of work per instruction).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2^x (hardware approximation, flushes subnormal results)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A softmax warp's part of the S row (ATT_KW columns) from TMEM.
__device__ __forceinline__ void attn_ld_part(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }
__device__ __forceinline__ void attn_ld_part(uint32_t taddr, float (&v)[64]) { tmem_ld64(taddr, v); }
// The same part of the P row as BF16 pairs (key 2i in the low half) into TMEM.
__device__ __forceinline__ void attn_st_p(uint32_t taddr, const float (&p)[32]) {
  float pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(p[2 * i], p[2 * i + 1]);
    pk[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&b2));
  }
  tmem_st16(taddr, pk);
}
__device__ __forceinline__ void attn_st_p(uint32_t taddr, const float (&p)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(p[2 * i], p[2 * i + 1]);
    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  tmem_st32(taddr, pk);
}

__global__ void __launch_bounds__(ATT_THREADS, 1)
    flash_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_vt, const AttnArgs args) {
  using C = AttnCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                   // [2] query tiles
  uint8_t* sK = sQ + C::Q_STAGES * C::Q_BYTES;
  uint8_t* sV = sK + C::K_STAGES * C::K_BYTES;
  float* xch = reinterpret_cast<float*>(sV + C::V_STAGES * C::V_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + C::V_STAGES * C::V_BYTES + C::XCH_BYTES);
  uint64_t* q_full = bars + 0;        // [Q_STAGES], by item
  uint64_t* q_empty = bars + 2;       // [2]: the item's S MMAs are done with its Q
  uint64_t* k_full = bars + 4;        // [K_STAGES <= 3]
  uint64_t* k_empty = bars + 7;       // [K_STAGES]
  uint64_t* v_full = bars + 10;       // [2]
  uint64_t* v_empty = bars + 12;      // [2]
  // Per S buffer b: s_full[b] / p_full[b] complete once per tile t (numbered
  // across items) with t % 3 == b. Neither can run two phases ahead of its
  // waiter: S_{t+3} is issued (with P_{t+1} V_{t+1}, or with the next item's
  // first tiles) only after P_{t+1} or P_t exist, hence after the softmax has
  // consumed S_t.
  uint64_t* s_full = bars + 14;       // [3]
  uint64_t* p_full = bars + 17;       // [3]
  uint64_t* o_done = bars + 20;       // [2]: P_t V_t done, tiles of parity t & 1
  uint64_t* o_free = bars + 22;       // the softmax warps have read an item's O
  uint64_t* mma_done = bars + 23;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::Q_STAGES; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < C::K_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&o_done[s], 1);
    }
    for (int s = 0; s < ATT_SBUF; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], ATT_SOFTMAX_WARPS);
    }
    mbar_init(o_free, ATT_SOFTMAX_WARPS);
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

  if (warp == 0 || warp == ATT_VWARP) {
    // ------------------------------------------------------------ producers
    // (one warp each, so neither producer's waits hold the other back)
    const bool kp = warp == 0;              // Q and K tiles; else V^T tiles
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      const volatile int never = 0;
      const int NS = kp ? C::K_STAGES : C::V_STAGES;
      uint64_t* full = kp ? k_full : v_full;
      uint64_t* empty = kp ? k_empty : v_empty;
      int t = 0, n = 0;                     // tiles and items issued
      bool ok = true;
      for (int it = blockIdx.x; ok && it < args.n_items; it += gridDim.x) {
        int qt, h, j0, j1;
        attn_item(args, it, &qt, &h);
        attn_key_tiles(qt, args.T, args.window, &j0, &j1);
        const int g = h / (args.nq / args.nkv);
        if (kp) {
          const int qb = n % C::Q_STAGES;
          if (!mbar_wait_bounded(&q_empty[qb], ((n / C::Q_STAGES) & 1) ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            break;
          }
          const int qrow = h * args.Tp + qt * ATT_BQ;
          uint8_t* sq = sQ + qb * C::Q_BYTES;
          mbar_arrive_expect_tx(&q_full[qb], C::Q_BYTES);
          tma_load_2d(sq, &tm_q, &q_full[qb], 0, qrow, pol);
          tma_load_2d(sq + C::Q_BYTES / 2, &tm_q, &q_full[qb], 64, qrow, pol);
        }
        ++n;
        // K tiles or V^T tiles of this item, into the ring
        for (int j = j0; j < j1; ++j) {
          const int s = t % NS;
          if (!mbar_wait_bounded(&empty[s], ((t / NS) & 1) ^ 1u, tmo, abort_flag)) {
            gemm_fail(abort_flag);
            ok = false;
            break;
          }
          const int k0 = j * ATT_BK;
          mbar_arrive_expect_tx(&full[s], C::K_BYTES);
          if (kp) {
            uint8_t* st = sK + s * C::K_BYTES;
            tma_load_2d(st, &tm_k, &full[s], 0, g * args.Tp + k0, pol);
            tma_load_2d(st + C::K_BYTES / 2, &tm_k, &full[s], 64, g * args.Tp + k0, pol);
          } else {
            uint8_t* st = sV + s * C::V_BYTES;
            tma_load_2d(st, &tm_vt, &full[s], k0, g * ATT_D, pol);
            tma_load_2d(st + C::V_BYTES / 2, &tm_vt, &full[s], k0 + 64, g * ATT_D, pol);
          }
          ++t;
        }
      }
      // every load must land before the CTA exits: the last phase of each
      // ring stage and Q buffer that was filled
      for (int u = max(0, t - NS); u < t; ++u)
        if (!mbar_wait_bounded(&full[u % NS], (u / NS) & 1, tmo, &never)) gemm_fail(abort_flag);
      if (kp)
        for (int u = max(0, n - C::Q_STAGES); u < n; ++u)
          if (!mbar_wait_bounded(&q_full[u % C::Q_STAGES], (u / C::Q_STAGES) & 1, tmo, &never))
            gemm_fail(abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t dO = tmem_base + ATT_O_COL;
      bool ok = true;
      int t0 = 0, n = 0;                    // first tile of the item, items done
      for (int it = blockIdx.x; ok && it < args.n_items; it += gridDim.x, ++n) {
        int qt, h, j0, j1;
        attn_item(args, it, &qt, &h);
        attn_key_tiles(qt, args.T, args.window, &j0, &j1);
        const int ntiles = j1 - j0;
        const int qb = n % C::Q_STAGES;
        if (!mbar_wait_bounded(&q_full[qb], (n / C::Q_STAGES) & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dq = sdesc_k128(smem_u32(sQ + qb * C::Q_BYTES));
        const uint64_t dq1 = sdesc_k128(smem_u32(sQ + qb * C::Q_BYTES + C::Q_BYTES / 2));
        // S_t = Q K_t^T into S buffer t % 3 (eight K = 16 steps; with pv set,
        // each step alternates with one step of O += P V issued by pv(kk), so
        // two independent accumulators share the tensor pipe)
        auto issue_s = [&](int t, auto&& pv) -> bool {
          const int ks = t % C::K_STAGES;
          if (!mbar_wait_bounded(&k_full[ks], (t / C::K_STAGES) & 1, tmo, abort_flag)) return false;
          tc_fence_after();
          const uint32_t base = smem_u32(sK + ks * C::K_BYTES);
          const uint64_t dk = sdesc_k128(base), dk1 = sdesc_k128(base + C::K_BYTES / 2);
          const uint32_t dS = tmem_base + static_cast<uint32_t>((t % ATT_SBUF) * 128);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            pv(kk);
            const uint64_t a = (kk < 4 ? dq : dq1) + 2 * (kk & 3);
            const uint64_t b = (kk < 4 ? dk : dk1) + 2 * (kk & 3);
            mma_bf16_ss(dS, a, b, idesc, kk != 0);
          }
          return true;
        };
        auto no_pv = [](int) {};
        // S of the item's first two tiles; their buffers held P of tiles
        // t0 - 3 and t0 - 2, whose P V were issued before
        for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
          ok = issue_s(t0 + j, no_pv);
          if (ok) {
            mma_commit(&s_full[(t0 + j) % ATT_SBUF]);
            mma_commit(&k_empty[(t0 + j) % C::K_STAGES]);
          }
        }
        for (int j = 0; ok && j < ntiles; ++j) {
          const int t = t0 + j;
          const int vs = t % C::V_STAGES;
          if (!mbar_wait_bounded(&p_full[t % ATT_SBUF], (t / ATT_SBUF) & 1, tmo, abort_flag) ||
              !mbar_wait_bounded(&v_full[vs], (t / C::V_STAGES) & 1, tmo, abort_flag) ||
              (j == 0 && n > 0 && !mbar_wait_bounded(o_free, (n - 1) & 1, tmo, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O += P_t V_t: P_t from TMEM (keys 16kk.. in columns 8kk..), V_t^T
          // from shared memory (two 64-key blocks); the item's first
          // overwrites O (the previous item's O has been read: o_free)
          const uint32_t dP = tmem_base + static_cast<uint32_t>((t % ATT_SBUF) * 128);
          const uint32_t base = smem_u32(sV + vs * C::V_BYTES);
          const uint64_t dv = sdesc_k128(base), dv1 = sdesc_k128(base + C::V_BYTES / 2);
          auto pv = [&](int kk) {
            const uint64_t b = (kk < 4 ? dv : dv1) + 2 * (kk & 3);
            mma_bf16_ts(dO, dP + 8 * kk, b, idesc, (j | kk) != 0);
          };
          if (j + 2 < ntiles) {
            if (!issue_s(t + 2, pv)) {
              ok = false;
              break;
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) pv(kk);
          }
          mma_commit(&o_done[t & 1]);
          mma_commit(&v_empty[vs]);
          if (j + 2 < ntiles) {
            mma_commit(&s_full[(t + 2) % ATT_SBUF]);
            mma_commit(&k_empty[(t + 2) % C::K_STAGES]);
          }
        }
        // every S MMA of the item has been issued: its Q buffer is free once
        // they complete
        if (ok) mma_commit(&q_empty[qb]);
        t0 += ntiles;
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
    const int part = (warp - 2) >> 2;       // keys / O columns [KW part, KW part + KW)
    const int row = q * 32 + lane;          // query row within the tile
    const uint32_t lanebits = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(part * ATT_KW);
    const int bar_id = 1 + q;               // named barrier of this lane quarter's warps
    const float NEG = -1e30f;
    // global layers' query scale is already in q; logits to base 2 in one FMA
    const float c2 = args.scale * ATT_LOG2E;
    const uint64_t cc = f2_pack(c2, c2);
    bool ok = true;
    int t0 = 0;                             // first tile of the item
    for (int it = blockIdx.x; it < args.n_items; it += gridDim.x) {
      int qt, h, j0, j1;
      attn_item(args, it, &qt, &h);
      attn_key_tiles(qt, args.T, args.window, &j0, &j1);
      const int ntiles = j1 - j0;
      const int qi = qt * ATT_BQ + row;     // query index
      const int hi = min(qi, args.T - 1);   // visible keys of row qi: [lo, hi]
      const int lo = args.window > 0 ? qi - args.window + 1 : 0;
      float m = NEG, l = 0.f;               // base-2 units; l over this part's keys
      for (int j = 0; j < ntiles; ++j) {
        const int t = t0 + j;
        const int s = t & 1;                // exchange slots
        const int sb = t % ATT_SBUF;        // S / P buffer
        if (ok) {
          bool ready = false;
          if (lane == 0) ready = mbar_wait_bounded(&s_full[sb], (t / ATT_SBUF) & 1, tmo, abort_flag);
          ok = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
        }
        float sv[ATT_KW];
        float mt = -INFINITY;
        if (ok) {
          tc_fence_after();
          attn_ld_part(tmem_base + lanebits + sb * 128 + col0, sv);
          const int k0 = (j0 + j) * ATT_BK + part * ATT_KW;
          if (__any_sync(0xffffffffu, k0 < lo || k0 + ATT_KW - 1 > hi)) {
#pragma unroll
            for (int c = 0; c < ATT_KW; ++c) {
              const int kj = k0 + c;
              sv[c] = (kj >= lo && kj <= hi) ? sv[c] : -INFINITY;
            }
          }
          // raw maximum in eight independent partials (long dependency chains
          // would stall the scheduler)
          float mp[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mp[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
          for (int c = 16; c < ATT_KW; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) mp[i] = fmax3(mp[i], sv[c + i], sv[c + 8 + i]);
          }
          mt = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * c2;
        }
        // tile maximum over all parts of the row (-inf from a failed part),
        // through slots of this tile's parity: a partner's next write to them
        // (tile t + 2) comes after the barrier of tile t + 1 (or an item's
        // end), which this warp reaches only after reading. The barrier also
        // orders every warp's S reads before any P write.
        float* xs = xch + s * ATT_PARTS * ATT_BQ;
        xs[part * ATT_BQ + row] = mt;
        tc_fence_before();
        named_bar_sync(bar_id, 32 * ATT_PARTS);
        tc_fence_after();
#pragma unroll
        for (int o = 1; o < ATT_PARTS; ++o) mt = fmaxf(mt, xs[((part + o) % ATT_PARTS) * ATT_BQ + row]);
        if (!ok) continue;
        // lazy reference: move m only when this tile exceeds it by more than TAU2
        const float mn = mt > m + ATT_TAU2 ? mt : m;
        const float alpha = ex2_approx(m - mn);
        const uint64_t nm = f2_pack(-mn, -mn);
        uint64_t sp[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < ATT_KW; c += 2) {
          float a, b;
          f2_unpack(f2_fma(f2_pack(sv[c], sv[c + 1]), cc, nm), a, b);
          sv[c] = ex2_approx(a);
          sv[c + 1] = ex2_approx(b);
          sp[(c >> 1) & 3] = f2_add(sp[(c >> 1) & 3], f2_pack(sv[c], sv[c + 1]));
        }
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a, b;
          f2_unpack(sp[i], a, b);
          ps += a + b;
        }
        l = l * alpha + ps;
        m = mn;
        // the O row is rescaled only after the previous P V has completed.
        // o_done[b] completes once per tile of parity b. At tile t every P V
        // up to t - 2 has completed (S_t was issued with P_{t-2} V_{t-2}, or
        // after it for an item's first two tiles, and its s_full commit
        // covers every MMA issued before it) and P_{t+1} V_{t+1} cannot have,
        // so the phase of P_{t-1} V_{t-1} is the current or the last one of
        // o_done[(t-1)&1]: the parity wait is exact even when earlier tiles
        // skipped it. (An item's first tile has no O to rescale.)
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          bool od = false;
          if (lane == 0)
            od = mbar_wait_bounded(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, tmo, abort_flag);
          ok = __shfl_sync(0xffffffffu, od ? 1 : 0, 0) != 0;
          if (!ok) continue;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < ATT_KW; c += 16) {
            float o[16];
            tmem_ld16(tmem_base + lanebits + ATT_O_COL + col0 + c, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_st16(tmem_base + lanebits + ATT_O_COL + col0 + c, o);
          }
        }
        // this part of the P row as BF16 pairs (key 2i in the low half) into
        // columns [KW/2 part, KW/2 part + KW/2) of this tile's S buffer
        attn_st_p(tmem_base + lanebits + sb * 128 + part * (ATT_KW / 2), sv);
        tmem_wait_st();
        // P and the O rescale visible to the MMA
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      // end of the item: O / l times the gate sigmoid(gate logit) (FP32),
      // BF16; l summed over all parts. The gate row part is fetched and its
      // sigmoid taken before the wait for the item's last P V, so its global
      // loads overlap it. o_done of the last tile t0 + ntiles - 1: its
      // previous phase (tile t0 + ntiles - 3) completed before S of the last
      // tile could, and the next item's first P V waits for o_free below.
      const bool valid = qi < args.T;
      float gt[ATT_KW];
      if (valid) {
        const float4* g4 = reinterpret_cast<const float4*>(
            args.gate + static_cast<size_t>(qi) * args.gate_ld + static_cast<size_t>(h) * ATT_D + col0);
#pragma unroll
        for (int i = 0; i < ATT_KW / 4; ++i) {
          const float4 t4 = g4[i];
          gt[4 * i] = t4.x; gt[4 * i + 1] = t4.y; gt[4 * i + 2] = t4.z; gt[4 * i + 3] = t4.w;
        }
#pragma unroll
        for (int i = 0; i < ATT_KW; ++i) gt[i] = __fdividef(1.0f, 1.0f + __expf(-gt[i]));
      }
      const int tl = t0 + ntiles - 1;
      if (ok) {
        bool od = false;
        if (lane == 0) od = mbar_wait_bounded(&o_done[tl & 1], (tl >> 1) & 1, tmo, abort_flag);
        ok = __shfl_sync(0xffffffffu, od ? 1 : 0, 0) != 0;
      }
      // row sums through their own slots: a partner rewrites its slot only
      // at the next item's end, after the barriers of that item's tiles,
      // which this warp reaches only after reading
      float* xl = xch + 2 * ATT_PARTS * ATT_BQ;
      xl[part * ATT_BQ + row] = l;
      named_bar_sync(bar_id, 32 * ATT_PARTS);
      float lt = l;
#pragma unroll
      for (int o = 1; o < ATT_PARTS; ++o) lt += xl[((part + o) % ATT_PARTS) * ATT_BQ + row];
      if (ok) {
        tc_fence_after();
        const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
        const size_t ld = static_cast<size_t>(args.nq) * ATT_D;
        __nv_bfloat16* orow = args.out + static_cast<size_t>(qi) * ld + static_cast<size_t>(h) * ATT_D + col0;
#pragma unroll
        for (int c = 0; c < ATT_KW; c += 16) {
          float o[16];
          tmem_ld16(tmem_base + lanebits + ATT_O_COL + col0 + c, o);
          if (valid) {
            uint4 pk[2];
            __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              p2[i] = __floats2bfloat162_rn(o[2 * i] * inv_l * gt[c + 2 * i],
                                            o[2 * i + 1] * inv_l * gt[c + 2 * i + 1]);
            uint4* d4 = reinterpret_cast<uint4*>(orow + c);
            d4[0] = pk[0];
            d4[1] = pk[1];
          }
        }
      }
      // this warp's O columns have been read: the next item may overwrite O
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      t0 += ntiles;
    }
    if (!ok && lane == 0) gemm_fail(abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace beam
