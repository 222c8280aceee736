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
#include <cuda_fp8.h>
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

}  // namespace beam
