// MXFP8 block quantisation helpers shared by the quantiser kernels and the GEMM epilogue.
// One UE8M0 scale 2^s per 32 elements, s the smallest integer with amax <= 448 * 2^s
// (s in [-127, 127]; an all-zero block takes s = -127); values times 2^-s are rounded to the
// nearest E4M3 value (ties to even) with saturation to +-448 by cvt.rn.satfinite.
#pragma once

#include "mok_device.cuh"

namespace mok {

// Scale-factor atoms.  The UE8M0 scales of 128 rows x one 128-element K block (4 bytes per row,
// one per 32 elements) are kept as 512 contiguous bytes with row r at byte 16 (r % 32) + 4 (r / 32)
// and block j of the 128 at + j: the shared-memory image that tcgen05.cp (32x128b, warpx4) moves
// into TMEM for the block-scaled MMA, so that a GEMM stage fetches each operand's scales with one
// bulk copy.  A scale tensor of rows x K/32 bytes is stored as [row tiles][K/128] atoms.
// Byte offset of the 4-byte word of row r (0..127) of row tile `tile` in K block kb of nkb.
__host__ __device__ __forceinline__ int64_t sf_atom_word(int64_t tile, int kb, int nkb, int r) {
  return (tile * nkb + kb) * 512 + 16 * (r & 31) + 4 * (r >> 5);
}

// Scale exponent of a block from its amax (fp32, finite, >= 0), by exact bit inspection:
// with amax = m 2^E, m in [1,2), the smallest s with amax <= 448 * 2^s = 1.75 * 2^(s+8) is
// E - 8 when m <= 1.75 and E - 7 otherwise.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = (int)((b >> 23) & 0xFF);
  if (ef == 0) return -127;  // zero or subnormal: 448 * 2^-127 exceeds every subnormal
  const uint32_t man = b & 0x7FFFFFu;
  // 448 = 1.75 * 2^8: amax <= 448 * 2^(e-8) iff the mantissa is <= 1.75
  int s = (ef - 127) - 8 + (man > 0x600000u ? 1 : 0);
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// Two fp32 values -> two E4M3 codes (lo at the lower byte).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantises 32 fp32 values of one block in registers: writes 32 codes (8 x uint32) and returns
// the scale byte.
__device__ __forceinline__ uint32_t mx_block32(const float (&v)[32], uint32_t (&q)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - s) << 23);  // 2^-s, s in [-127, 126]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    const uint32_t b = e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    q[i] = a | (b << 16);
  }
  return (uint32_t)(s + 127);
}

}  // namespace mok
