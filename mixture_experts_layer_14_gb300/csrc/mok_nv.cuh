// NVFP4 helpers shared by the quantiser kernels (nv.cu) and the GEMM's NVFP4 modes.
//
// Format: NVIDIA's NVFP4 (the first page names it as the format of its authors' earlier
// kernels): E2M1 elements (sign, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0, 0.5,
// 1, 1.5, 2, 3, 4, 6), one E4M3 scale per 16 consecutive elements along the reduction
// dimension, one fp32 scale per tensor.  Recipe, every step an fp32 operation rounded to nearest
// even: S = 2688 / A for the tensor amax A (1 when A is 0); a block of amax a takes the scale
// s = E4M3_rn((a / 6) * S) (saturating); an element v the code E2M1_rn(v * (S / s)) (ties to the
// even code, saturating at 6; 0 when s is 0; sign bit when v * (S / s) < 0).  The value is
// q * s / S: products q * s are exact in f16, and 1 / S is applied in the GEMM epilogue.
#pragma once

#include <cuda_fp16.h>

#include "mok_mx.cuh"

namespace mok {

constexpr float kNvRange = 2688.0f;  // 6 * 448

__device__ __forceinline__ float nv_tensor_S(float amax) {
  return amax > 0.0f ? __fdiv_rn(kNvRange, amax) : 1.0f;
}
// the tensor's decode scale 1 / S
__device__ __forceinline__ float nv_decode_g(float amax) { return __fdiv_rn(1.0f, nv_tensor_S(amax)); }

// (s, s) as f16x2 for an E4M3 code s (exact: every E4M3 value is an f16 value)
__device__ __forceinline__ uint32_t e4m3_bcast_f16x2(uint32_t code) {
  uint32_t r;
  const uint16_t c2 = (uint16_t)(code | (code << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c2));
  return r;
}
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  return __half2float(__ushort_as_half((unsigned short)(e4m3_bcast_f16x2(code) & 0xFFFFu)));
}

// Eight E2M1 codes (one 32-bit word; element 2j in the low nibble of byte j, 2j + 1 in its high
// nibble) -> four f16x2 words, element 2j in the low half of word j.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

struct NvScale {
  uint32_t code;  // E4M3 code of the block scale
  float val;      // its value
  float inv;      // S / val (0 when val is 0)
};
__device__ __forceinline__ NvScale nv_block_scale(float amax, float S) {
  NvScale b;
  const float u = __fmul_rn(__fdiv_rn(amax, 6.0f), S);
  b.code = e4m3x2(u, 0.0f) & 0xFFu;
  b.val = e4m3_value(b.code);
  b.inv = b.val > 0.0f ? __fdiv_rn(S, b.val) : 0.0f;
  return b;
}

// E2M1 code of v in a block of scale b: the magnitude index by comparisons with the midpoints
// of the grid (ties to the even index: 0.25 -> 0, 0.75 -> 2, 1.25 -> 2, 1.75 -> 4, 2.5 -> 4,
// 3.5 -> 6, 5 -> 6), saturating at 6.
__device__ __forceinline__ uint32_t nv_code(float v, const NvScale& b) {
  const float t = __fmul_rn(v, b.inv);
  const float a = fabsf(t);
  const uint32_t idx = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                       (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                       (uint32_t)(a > 5.0f);
  return idx | (t < 0.0f ? 8u : 0u);
}
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t i = code & 7u;
  const float m = i <= 4u ? 0.5f * (float)i : (i == 7u ? 6.0f : (float)(i - 2u));
  return (code & 8u) ? -m : m;
}

// A block of 16 fp32 values -> 8 f16x2 words of their NVFP4 values without the tensor scale
// (q * s, exact in f16).
__device__ __forceinline__ void nv_block16_values(const float* v, float S, uint32_t* out) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  const NvScale b = nv_block_scale(a, S);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lo = e2m1_value(nv_code(v[2 * i], b)) * b.val;
    const float hi = e2m1_value(nv_code(v[2 * i + 1], b)) * b.val;
    const __half2 h = __halves2half2(__float2half_rn(lo), __float2half_rn(hi));
    out[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

}  // namespace mok
