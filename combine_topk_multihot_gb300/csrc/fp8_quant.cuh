// Rowwise e4m3 quantization of bf16 rows, shared by the FP8 row kernels and
// the fused dispatch's FP8 rows.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds, scope note: FP8 dispatch is the named follow-up.
// Format: one fp32 scale per row, scale = amax(|row|) / 448 (1 for an
// all-zero row), code = e4m3(v / scale) rounded to nearest even and saturated
// at +-448, the division an IEEE fp32 division.  A warp owns a row: lane l
// holds the 8-value (16-byte) vectors l, l + 32, ...
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

constexpr float E4M3_MAX = 448.0f;

__device__ __forceinline__ float bf16_abs_max8(uint4 q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  return m;
}

__device__ __forceinline__ uint32_t e4m3_of(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// 8 bf16 values / scale -> 8 e4m3 codes, in element order (lowest byte first).
__device__ __forceinline__ uint2 quantize8(uint4 q, float scale) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = e4m3_of(bf16_lo(w[i]) / scale) | (e4m3_of(bf16_hi(w[i]) / scale) << 8);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// The scale of a warp-owned row (V vectors per lane).
__device__ __forceinline__ float row_scale(const uint4* src, int V, int lane) {
  float amax = 0.f;
  for (int v = 0; v < V; ++v) amax = fmaxf(amax, bf16_abs_max8(__ldg(src + lane + 32 * v)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, o));
  return amax > 0.f ? amax / E4M3_MAX : 1.0f;
}

}  // namespace moe
