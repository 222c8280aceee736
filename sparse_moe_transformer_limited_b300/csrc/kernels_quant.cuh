// Per-row E4M3 quantisation for the FP8 expert weights and activations.
//
// "Reflection 放出 501B 的 Beam 权重：四套精度、滑动窗口和一场榜单落差", section
// 四套权重的账，自己算一遍: the FP8 checkpoint stores the linear weights as
// F8_E4M3 and is a dynamic FP8 quantisation (activation scales computed at
// run time). One FP32 scale per row:
//   amax = max_j |v_j|;  scale = amax / 448;  inv = 448 / amax   (FP32, IEEE
//   division; scale = inv = 1 for a zero row)
//   code_j = E4M3(v_j * inv)   (the FP32 product, then round to nearest even,
//                                saturating at +-448)
// and a row is dequantised as E4M3 value * scale. The same kernel quantises
// weight rows (once, offline), the expert input x per token (gathering the
// rows into expert order on the way) and the SwiGLU output per pair.
//
// One warp per row; 16-byte loads of 8 BF16 values, 8-byte stores of 8 codes.
// Bound by HBM bandwidth (2 bytes read and 1 written per element; the second
// read of the row for the codes hits L1/L2).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace beam {

constexpr float kE4M3Max = 448.0f;

// dst row r = quantised src row (src_row ? src_row[r] : r); K % 8 == 0.
__global__ void __launch_bounds__(256) quant_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ src,
                                                              const int* __restrict__ src_row,
                                                              long long rows, int K,
                                                              uint8_t* __restrict__ dst,
                                                              float* __restrict__ dst_scale) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const long long sr = src_row ? src_row[r] : r;
  const uint4* s = reinterpret_cast<const uint4*>(src + sr * K);
  const int nc = K >> 3;
  float amax = 0.f;
  for (int c = lane; c < nc; c += 32) {
    const uint4 v = s[c];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const bool nz = amax > 0.f;
  const float inv = nz ? __fdiv_rn(kE4M3Max, amax) : 1.f;
  if (lane == 0) dst_scale[r] = nz ? __fdiv_rn(amax, kE4M3Max) : 1.f;
  uint2* d = reinterpret_cast<uint2*>(dst + r * K);
  for (int c = lane; c < nc; c += 32) {
    const uint4 v = s[c];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      const uint32_t c0 = __nv_cvt_float_to_fp8(__fmul_rn(f.x, inv), __NV_SATFINITE, __NV_E4M3);
      const uint32_t c1 = __nv_cvt_float_to_fp8(__fmul_rn(f.y, inv), __NV_SATFINITE, __NV_E4M3);
      // element 2i in byte (2i % 4), element 2i+1 in the next byte (little endian)
      w[i >> 1] |= (c0 | (c1 << 8)) << (16 * (i & 1));
    }
    d[c] = make_uint2(w[0], w[1]);
  }
}


// ---------------------------------------------------------------------------
// NVFP4 ("Reflection 放出 501B 的 Beam 权重…", section 四套权重的账，自己算一遍:
// every routed-expert weight packed as two 4-bit values per byte; section
// 上手前的五个坑: the FP4 tensor-core path of Blackwell). E2M1 elements, one
// E4M3 block scale per 16 elements along K and one FP32 scale per group of
// rows (an expert matrix, or one activation row). In FP32, IEEE division:
//   g   = amax_group / 2688            (2688 = 6 * 448; g = 1 for amax 0)
//   s_b = E4M3(amax_b / (6 * g))       (round to nearest even, saturating)
//   q_i = E2M1(v_i * (1 / (s_b * g)))  (round to nearest even, saturating
//                                       at 6; q = 0 where s_b = 0)
// Codes: two per byte, the even element in the low nibble. Block scales are
// stored in 512-byte groups, one per (tile of `tile` rows, K = 64 step),
// tile = 128 (weights; the MMA's M) or the token tile (32 or 128):
//   group (r / tile) * (K / 64) + k / 64,
//   byte (r % 32) * 16 + ((r % tile) / 32) * 4 + (k % 64) / 16
// -- the layout the tensor cores read after a 32x128b.warpx4 copy to TMEM,
// each token tile's scales starting at its group's first column.
// ---------------------------------------------------------------------------
constexpr float kNvfp4GroupDiv = 2688.0f;

__device__ __forceinline__ size_t nvfp4_sf_index(long long r, int K, int blk, int tile) {
  return (static_cast<size_t>(r / tile) * (K >> 6) + (blk >> 2)) * 512 +
         static_cast<size_t>((r & 31) * 16 + ((r % tile) >> 5) * 4 + (blk & 3));
}

// Largest magnitude in each group of rows_per_group consecutive rows, as the
// bits of a non-negative float (so atomicMax orders them). `gmax` must be
// zero on entry. One warp per row.
__global__ void __launch_bounds__(256) group_amax_kernel(const __nv_bfloat16* __restrict__ src,
                                                         long long rows, int K, int rows_per_group,
                                                         unsigned* __restrict__ gmax) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* s = reinterpret_cast<const uint4*>(src + r * K);
  float amax = 0.f;
  for (int c = lane; c < (K >> 3); c += 32) {
    const uint4 v = s[c];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) atomicMax(gmax + r / rows_per_group, __float_as_uint(amax));
}

// gscale[i] = g of group i from its largest magnitude (held as bits in the same array).
__global__ void nvfp4_group_scale_kernel(float* __restrict__ gscale, long long groups) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= groups) return;
  const float amax = __uint_as_float(reinterpret_cast<const unsigned*>(gscale)[i]);
  gscale[i] = amax > 0.f ? __fdiv_rn(amax, kNvfp4GroupDiv) : 1.f;
}

// NVFP4 quantisation of rows, one warp per row r < min(rows, *rows_dev):
// source row src_row ? src_row[r] : r; a row with row_valid[r] < 0 becomes
// zero codes and zero block scales (and scale 1). Per-row groups when
// gmax == nullptr (gscale[r] written here); else the group maxima come from
// gmax (as bits) and gscale is not written. K % 64 == 0; sf_tile = 32 or
// 128 (rows per block-scale tile).
__global__ void __launch_bounds__(256) quant_rows_nvfp4_kernel(
    const __nv_bfloat16* __restrict__ src, const int* __restrict__ src_row,
    const int* __restrict__ row_valid, long long rows, const int* __restrict__ rows_dev, int K,
    int rows_per_group, const unsigned* __restrict__ gmax, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, float* __restrict__ gscale, int sf_tile) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long limit = rows_dev ? min(rows, static_cast<long long>(*rows_dev)) : rows;
  if (r >= limit) return;
  const int nblk = K >> 4;
  uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
  if (row_valid != nullptr && row_valid[r] < 0) {
    for (int b = lane; b < nblk; b += 32) {
      crow[b] = make_uint2(0u, 0u);
      sf[nvfp4_sf_index(r, K, b, sf_tile)] = 0;
    }
    if (gmax == nullptr && lane == 0) gscale[r] = 1.f;
    return;
  }
  const long long sr = src_row ? src_row[r] : r;
  const uint4* s = reinterpret_cast<const uint4*>(src + sr * K);
  float amax;
  if (gmax != nullptr) {
    amax = __uint_as_float(gmax[r / rows_per_group]);
  } else {
    amax = 0.f;
    for (int c = lane; c < (K >> 3); c += 32) {
      const uint4 v = s[c];
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  const float g = amax > 0.f ? __fdiv_rn(amax, kNvfp4GroupDiv) : 1.f;
  if (gmax == nullptr && lane == 0) gscale[r] = g;
  const float six_g = __fmul_rn(6.f, g);
  for (int b = lane; b < nblk; b += 32) {
    float v[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 w = s[2 * b + h];
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        v[8 * h + 2 * i] = f.x;
        v[8 * h + 2 * i + 1] = f.y;
      }
    }
    float amax_b = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(v[i]));
    const __nv_fp8_storage_t sb =
        __nv_cvt_float_to_fp8(__fdiv_rn(amax_b, six_g), __NV_SATFINITE, __NV_E4M3);
    const float sbv = __half2float(__half(__nv_cvt_fp8_to_halfraw(sb, __NV_E4M3)));
    const float inv = sbv > 0.f ? __fdiv_rn(1.f, __fmul_rn(sbv, g)) : 0.f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t q =
          static_cast<uint32_t>(__nv_cvt_float_to_fp4(__fmul_rn(v[i], inv), __NV_E2M1, cudaRoundNearest)) & 0xFu;
      w[i >> 3] |= q << (4 * (i & 7));   // element i: nibble i % 8 of word i / 8
    }
    crow[b] = make_uint2(w[0], w[1]);
    sf[nvfp4_sf_index(r, K, b, sf_tile)] = static_cast<uint8_t>(sb);
  }
}

}  // namespace beam
