// The router-weighted combine, post-RMSNorm and scaled residual, fused into
// the epilogue of the down-projection GEMMs ("Reflection 发布 Beam 501B 开源模型，
// 支持 1M tokens 上下文", section 专家混合模型: the expert outputs of a token are
// summed with its normalised router weights; section 残差流: the sublayer
// output is normalised, then h_k = sqrt((k-1)/k) * h_{k-1} + (1/sqrt(k)) * n,
// in FP32).
//
// Each epilogue adds c_r * y_r[h] for its (pair row r, hidden column h)
// elements into an FP32 accumulator o[t, h] of the pair's token t with an
// L2 reduction (red.global.add), c_r = the pair's router weight times the
// activation row scale of the quantised paths. Once a warp (or a lane) has
// added its share for a token it counts one arrival on that token's counter;
// the arrival that completes the token's count (`expected`, fixed by the
// kernel's tiling: every token receives the same number) appends the token
// to a completion list. Completions bunch up at the end of the GEMM (a token
// is done when the last of its experts is), so finalising them where they
// complete would stall a few epilogues; instead every epilogue warp of the
// grid, once its own units are done, takes list entries in order and
// finalises those rows:
//   resid:  out[t] = bf16( a * h_prev[t] + b * RMSNorm(o[t]) * gain )
//   else:   out[t] = o[t]  (bf16, or fp32 with out_f32)
// The adds land in a different order from run to run, so o (and the output)
// is reproducible to FP32 rounding, not bitwise.
//
// Ordering: every thread fences (gpu scope) after its adds and before the
// warp's counter increments; the completing lane fences before it publishes
// the token in the list; the finalising warp fences after it reads the entry
// and reads o through L2 (ld.global.cg). The accumulator, the counters and
// the list must be cleared before the GEMM starts (clear_acc_kernel). Every
// wait for a list entry is bounded.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels_rows.cuh"
#include "ptx.cuh"

namespace beam {

struct CombineArgs {
  float* acc;               // o [T, H] FP32, zero on entry
  int* count;               // [T] arrivals per token, zero on entry
  int* done;                // [T] completed tokens in completion order, -1 on entry
  int* cursor;              // [2] {list entries written, entries taken}, zero on entry
  int T;
  int expected;             // arrivals that complete one token
  const int* row_token;     // [rows] token of each expert-ordered row (-1: padding)
  const float* row_weight;  // [rows] router weight of each row
  const float* row_scale;   // [rows] activation row scale (quantised paths) or NULL
  const __nv_bfloat16* h_prev;  // [T, H] residual input (resid)
  const float* gain;        // [H] post-norm gain or NULL (= 1)
  void* out;                // [T, H] bf16 (or fp32 when out_f32)
  int H;
  float eps, a, b;
  int resid;
  int out_f32;
  // 0: per-token arrival counters and the completion list (above); else
  // every epilogue warp of the grid counts itself done once after all its
  // units, and once all have, the warps finalise the T tokens between them
  // (combine_grid_finish; the weight-major kernel, where tokens are few)
  int grid_done;
};

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4_f32(float* p, float x, float y, float z, float w) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x),
               "f"(y), "f"(z), "f"(w)
               : "memory");
}

// Coefficient of an expert-ordered row: router weight x activation row scale
// (0 for a padding row, whose adds are skipped by the callers).
__device__ __forceinline__ float combine_coef(const CombineArgs& c, int r) {
  const float w = c.row_weight[r];
  return c.row_scale != nullptr ? w * c.row_scale[r] : w;
}

// One warp finalises token t (all 32 lanes take part): two passes over the
// FP32 row through L2 with many 16-byte loads in flight per lane (the row is
// 4H bytes; H <= 8192).
__device__ __noinline__ void combine_finalize_token(const CombineArgs& c, int t, int lane) {
  const int H = c.H;
  const float4* o = reinterpret_cast<const float4*>(c.acc + static_cast<size_t>(t) * H);
  const int nc = H >> 3;   // 8-element chunks
  float r = 1.f;
  if (c.resid) {
    float ss = 0.f;
    const int n4 = H >> 2;
#pragma unroll 16
    for (int k = lane; k < n4; k += 32) {
      const float4 p = __ldcg(o + k);
      ss = fmaf(p.x, p.x, ss); ss = fmaf(p.y, p.y, ss); ss = fmaf(p.z, p.z, ss); ss = fmaf(p.w, p.w, ss);
    }
    ss = warp_sum(ss);
    r = rsqrtf(ss / static_cast<float>(H) + c.eps);
  }
#pragma unroll 8
  for (int k = lane; k < nc; k += 32) {
    const float4 p = __ldcg(o + 2 * k);
    const float4 q = __ldcg(o + 2 * k + 1);
    if (c.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(c.out) + static_cast<size_t>(t) * H) + 2 * k;
      dst[0] = p;
      dst[1] = q;
      continue;
    }
    float f[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
    if (c.resid) {
      float hv[8], g[8];
      load8(c.h_prev + static_cast<size_t>(t) * H, k, hv);
      gain8(c.gain, k, g);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = fmaf(c.a, hv[e], c.b * (f[e] * r * g[e]));
    }
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(c.out) + static_cast<size_t>(t) * H)[k] =
        f32x8_to_bf16(f);
  }
}

// Called by a whole warp after its adds for up to 32 * NT tokens: lane j
// counts one arrival for each of its tokens tok[i] (< 0: none); a lane whose
// arrival completes a token appends it to the completion list. One fence
// covers all of the warp's adds.
template <int NT>
__device__ __forceinline__ void combine_arrive_warp(const CombineArgs& c, const int (&tok)[NT]) {
  __threadfence();
  __syncwarp();
  bool last[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i)
    last[i] = tok[i] >= 0 && atomicAdd(c.count + tok[i], 1) == c.expected - 1;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    if (last[i]) {
      __threadfence();
      const int pos = atomicAdd(c.cursor, 1);
      asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(c.done + pos), "r"(tok[i]) : "memory");
    }
  }
}
__device__ __forceinline__ void combine_arrive_warp(const CombineArgs& c, int tok, int lane) {
  const int t1[1] = {tok};
  combine_arrive_warp<1>(c, t1);
}

// Called by a whole warp once its own units are done: takes list entries in
// order until all T tokens are taken, waits (bounded by timeout_ns, or until
// `abort_flag` is set) for each entry to be published and finalises its row.
// Returns false on a timeout.
__device__ __forceinline__ bool combine_drain_warp(const CombineArgs& c, int lane,
                                                   unsigned long long timeout_ns,
                                                   const volatile int* abort_flag) {
  while (true) {
    int i = 0;
    if (lane == 0) i = atomicAdd(c.cursor + 1, 1);
    i = __shfl_sync(0xffffffffu, i, 0);
    if (i >= c.T) return true;
    int t = -1;
    if (lane == 0) {
      const unsigned long long t0 = globaltimer_ns();
      while (true) {
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(t) : "l"(c.done + i) : "memory");
        if (t >= 0 || *abort_flag || globaltimer_ns() - t0 > timeout_ns) break;
        __nanosleep(256);
      }
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t < 0) return false;
    __threadfence();
    combine_finalize_token(c, t, lane);
  }
}

// Grid-wide completion (grid_done): called by every epilogue warp of the
// grid once its own units are done; warp wid of nwarps finalises tokens wid,
// wid + nwarps, ... after all nwarps warps have counted themselves in
// cursor[0] (each after a fence that covers its reductions). The wait is
// bounded; returns false on a timeout. Every CTA of the grid is resident
// (one per SM), as the completion list's waits also assume.
__device__ __forceinline__ bool combine_grid_finish(const CombineArgs& c, int lane, int wid,
                                                    int nwarps, unsigned long long timeout_ns,
                                                    const volatile int* abort_flag) {
  __threadfence();
  __syncwarp();
  int n = 0;
  if (lane == 0) {
    atomicAdd(c.cursor, 1);
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(n) : "l"(c.cursor) : "memory");
      if (n >= nwarps || *abort_flag || globaltimer_ns() - t0 > timeout_ns) break;
      __nanosleep(256);
    }
  }
  n = __shfl_sync(0xffffffffu, n, 0);
  if (n < nwarps) return false;
  __threadfence();
  for (int t = wid; t < c.T; t += nwarps) combine_finalize_token(c, t, lane);
  return true;
}

// Before the down GEMM: o = 0 (n4 float4), counters = 0, list entries = -1,
// cursors = 0.
__global__ void __launch_bounds__(256) clear_acc_kernel(float4* __restrict__ acc, size_t n4,
                                                        int* __restrict__ count,
                                                        int* __restrict__ done,
                                                        int* __restrict__ cursor, int T) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < n4; i += stride) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = i0; i < static_cast<size_t>(T); i += stride) {
    count[i] = 0;
    done[i] = -1;
  }
  if (i0 < 2) cursor[i0] = 0;
}

}  // namespace beam
