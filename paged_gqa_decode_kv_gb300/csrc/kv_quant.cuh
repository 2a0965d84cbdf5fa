// kv_quant.cuh -- the 8-bit cache's quantisation of one K or V row, shared by
// the kernels that append into an 8-bit pool (kv_append.cu and the fused
// append of short_attention.cu), so that every path writes the same bits.
//
// "Ch. 6 Inference efficiency and serving", 6.6.1: symmetric quantisation
// with the scale from the largest absolute value (a zero row takes a positive
// scale); "The math of Transformer inference", section 11: KV scales per head
// and per token.  For a row x of 128 bf16 values: scale = max|x| / 448 (1 if
// that is 0), code_i = E4M3(x_i / scale), both divisions IEEE binary32, the
// conversion rounding to nearest even and saturating to +-448.
#pragma once

#include <cuda_fp8.h>

#include "pgd_device.cuh"

namespace pgd {

constexpr int kGroupBytes8 = 8 * kHeadDim + 32;  // an 8-token group: codes, then 8 scales

// Called by all 32 lanes of a warp; each 16-lane half quantises one row,
// lane l of the half holding dims 8 l .. 8 l + 7 in `raw`.  Returns that
// lane's 8 codes (two words, dims in order) and the half's row scale.
__device__ __forceinline__ void quantize_row_e4m3(const uint4 &raw, uint32_t (&w)[2],
                                                  float &scale) {
  float f[8];
  unpack8(raw, f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
  scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint16_t c0 = (uint16_t)__nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[4 * j], scale), __fdiv_rn(f[4 * j + 1], scale)), __NV_SATFINITE,
        __NV_E4M3);
    const uint16_t c1 = (uint16_t)__nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[4 * j + 2], scale), __fdiv_rn(f[4 * j + 3], scale)),
        __NV_SATFINITE, __NV_E4M3);
    w[j] = (uint32_t)c0 | ((uint32_t)c1 << 16);
  }
}

// Where lane l's 8 codes of token slot s go inside the slot's 8-token group
// (dims 8 l .. 8 l + 7: core matrix l / 2, half l % 2), and the slot's scale.
__device__ __forceinline__ int code_offset8(int slot, int l) {
  return (l >> 1) * 128 + (slot & 7) * 16 + (l & 1) * 8;
}
__device__ __forceinline__ int scale_offset8(int slot) { return 8 * kHeadDim + (slot & 7) * 4; }

// Two E4M3 codes (x.x in the low byte) widened to binary32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
  const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3));
  return __half22float2(h);
}

}  // namespace pgd
