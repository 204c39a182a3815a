// NVFP4 quantisers of the layer's NVFP4 variant (format and recipe in mok_nv.cuh): the weights
// once (per-matrix amax, then codes and block scales in the GEMM's operand layout), the
// activation x per forward with its calibrated tensor amax, and the calibration setter.
#include "mok_nv.cuh"

namespace mok {

// amax[m] = max |src[m]| over each of nmat matrices of `per` bf16 elements (a multiple of 8):
// an atomicMax of the bit pattern, which orders non-negative floats like their values.
__global__ void __launch_bounds__(256) nv_amax_kernel(const __nv_bfloat16* __restrict__ src,
                                                      int64_t per, uint32_t* __restrict__ amax) {
  const int m = blockIdx.y;
  const uint4* p = reinterpret_cast<const uint4*>(src + (int64_t)m * per);
  float a = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per / 8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 u = p[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  __shared__ float s_a[8];
  if ((threadIdx.x & 31) == 0) s_a[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) a = fmaxf(a, s_a[i]);
    atomicMax(amax + m, __float_as_uint(a));
  }
}

// Weights src [nmat][K][N] bf16 (the layer's x @ W layout) -> for every (matrix, 64-element K
// block kb, column n) a row of 32 code bytes (byte j: elements 2j and 2j + 1 of the block, low
// nibble first) at q[((m K/64 + kb) N + n) 32] and a row of 4 scale bytes (one per 16 elements)
// at sc[((m K/64 + kb) N + n) 4]; g[m] = 1 / S of the matrix.  One thread per (matrix, 16-element
// K block, column): 16 strided reads, coalesced across the warp.
__global__ void __launch_bounds__(256) nv_quantize_weight_kernel(
    const __nv_bfloat16* __restrict__ src, int64_t nmat, int K, int N,
    const uint32_t* __restrict__ amax, uint8_t* __restrict__ q, uint8_t* __restrict__ sc,
    float* __restrict__ g) {
  const int nb = K / 16;
  const int64_t total = nmat * (int64_t)nb * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int n = (int)(i % N);
    const int64_t rest = i / N;
    const int b = (int)(rest % nb);
    const int64_t m = rest / nb;
    const float S = nv_tensor_S(__uint_as_float(amax[m]));
    const __nv_bfloat16* col = src + (m * K + 16 * b) * N + n;
    float v[16];
    float a = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      v[r] = __bfloat162float(col[(int64_t)r * N]);
      a = fmaxf(a, fabsf(v[r]));
    }
    const NvScale s = nv_block_scale(a, S);
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      lo |= nv_code(v[r], s) << (4 * r);
      hi |= nv_code(v[8 + r], s) << (4 * r);
    }
    const int64_t row = (m * (K / 64) + b / 4) * N + n;
    *reinterpret_cast<uint2*>(q + row * 32 + 8 * (b & 3)) = make_uint2(lo, hi);
    sc[row * 4 + (b & 3)] = (uint8_t)s.code;
    if (n == 0 && b == 0) g[m] = __fdiv_rn(1.0f, S);
  }
}

// rows x K bf16 -> rows x K f16, each block of 16 replaced by its NVFP4 values without the tensor
// scale (q * s), with the tensor amax *amax (a calibrated value).  One thread per block.
__global__ void __launch_bounds__(256) nv_quantize_act_kernel(const __nv_bfloat16* __restrict__ src,
                                                              int64_t nblocks,
                                                              const float* __restrict__ amax,
                                                              __half* __restrict__ dst) {
  const float S = nv_tensor_S(*amax);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + 16 * i);
    float v[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = s4[h];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * h + 2 * j] = bf16_lo(w[j]);
        v[8 * h + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
    uint32_t o[8];
    nv_block16_values(v, S, o);
    uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * i);
    d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

__global__ void nv_set_act_kernel(float* act, float amax_x, float amax_h) {
  act[0] = amax_x;
  act[1] = amax_h;
}

cudaError_t launch_nv_prepare(const void* src, int64_t nmat, int K, int N, uint32_t* amax, void* q,
                              void* sc, float* g, cudaStream_t s) {
  if (nmat == 0) return cudaSuccess;
  const int64_t per = (int64_t)K * N;
  const int bx = (int)std::min<int64_t>((per / 8 + 255) / 256, 64);
  prof_begin("nv_amax", s);
  nv_amax_kernel<<<dim3(bx, (unsigned)nmat), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), per, amax);
  prof_end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t total = nmat * (int64_t)(K / 16) * N;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 16);
  prof_begin("nv_quantize_weight", s);
  nv_quantize_weight_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), nmat, K, N,
                                                        amax, static_cast<uint8_t*>(q),
                                                        static_cast<uint8_t*>(sc), g);
  prof_end(s);
  return cudaGetLastError();
}

cudaError_t launch_nv_quantize_act(const void* src, int64_t rows, int K, const float* amax,
                                   void* dst, cudaStream_t s) {
  const int64_t nblocks = rows * (int64_t)(K / 16);
  if (nblocks == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((nblocks + 255) / 256, (int64_t)num_sms() * 16);
  prof_begin("nv_quantize_x", s);
  nv_quantize_act_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), nblocks, amax,
                                                     static_cast<__half*>(dst));
  prof_end(s);
  return cudaGetLastError();
}

cudaError_t launch_nv_set_act(float* act, float amax_x, float amax_h, cudaStream_t s) {
  nv_set_act_kernel<<<1, 1, 0, s>>>(act, amax_x, amax_h);
  return cudaGetLastError();
}

}  // namespace mok
