// Bandwidth-bound kernels of the MoE layer: the pull gather of token rows into each expert's
// region, the fixed-order combine, and the router-weight backward.  One warp per row, 16-byte
// vector accesses, grid-stride loops over a grid of a few blocks per SM.
#include <type_traits>

#include "mok_device.cuh"

namespace mok {

constexpr int kRowThreads = 256;
constexpr int kCombineSplit = 2;

static int rows_grid(int64_t nrows) {
  const int64_t blocks = (nrows + (kRowThreads / 32) - 1) / (kRowThreads / 32);  // one warp per row
  return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms() * 8));
}

// Pull gather (page "Метод и эксперименты": each expert pulls its tokens' rows into its region):
// for every kept route (t, j), dst[inv_pos[t, j]] = src[t].  Token-major: each source row is read
// once and written to its k destination rows, so a source larger than L2 is read from memory
// once rather than once per route.  With a second source (the backward pulls x and dY with the
// same schedule) the warps take both in one list.  Rows are handled as 16-byte vectors (bf16
// rows and E4M3 code rows alike); destination rows that no kept route names are not written.
__global__ void __launch_bounds__(kRowThreads) gather_rows_kernel(
    const uint4* __restrict__ src0, const uint4* __restrict__ src1,
    const int32_t* __restrict__ inv_pos, int64_t T, int k, int vec_per_row,
    uint4* __restrict__ dst0, uint4* __restrict__ dst1) {
  const int lane = threadIdx.x & 31;
  const int64_t wglobal = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = src1 ? 2 * T : T;
  for (int64_t tt = wglobal; tt < total; tt += nwarps) {
    const bool second = tt >= T;
    const int64_t t = second ? tt - T : tt;
    const uint4* s = (second ? src1 : src0) + t * vec_per_row;
    uint4* dbase = second ? dst1 : dst0;
    const int mine = lane < k ? inv_pos[t * k + lane] : -1;  // lane j: destination of route j
    int dst_row[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) dst_row[j] = __shfl_sync(0xffffffffu, mine, j);
    // four 16-byte loads in flight per lane, each stored to every destination row with
    // evict-first stores (they are read back by the next kernel, not by this one)
    for (int v = lane; v < vec_per_row; v += 128) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v + 32 * u < vec_per_row) a[u] = s[v + 32 * u];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && dst_row[j] >= 0) {
          uint4* d = dbase + (int64_t)dst_row[j] * vec_per_row;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (v + 32 * u < vec_per_row) __stcs(d + v + 32 * u, a[u]);
        }
      }
    }
  }
}

cudaError_t launch_gather_rows(const char* name, const void* src0, const void* src1,
                               const int32_t* inv_pos, int64_t T, int k, int row_bytes,
                               void* dst0, void* dst1, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  prof_begin(name, s);
  gather_rows_kernel<<<rows_grid(src1 ? 2 * T : T), kRowThreads, 0, s>>>(
      static_cast<const uint4*>(src0), static_cast<const uint4*>(src1), inv_pos, T, k,
      row_bytes / 16, static_cast<uint4*>(dst0), static_cast<uint4*>(dst1));
  prof_end(s);
  return cudaGetLastError();
}

// y[t] = Ysh[t] (+ Ysh2[t]) + sum over the token's routes in ascending expert id of
// Ys[inv_pos[t,j]] (fp32 accumulation, one bf16 rounding; Ysh2 is the router term dl W_r^T of
// the MXFP8 backward's dX).  The router weight is already inside Ys (it is
// applied in the down-projection epilogue).  Page "Mixture-of-Kittens: Nhân kernel MoE ...",
// section "Chồng lấp tính toán ...": the layer combines shared and routed expert outputs with
// the router weights; the fixed order keeps the result bit-identical across runs.
// One instantiation per k (and per presence of Ysh2), so that the row loads of a vector are
// unconditional and all in flight together; a dropped route (inv_pos = -1) reads row 0 and is
// multiplied by zero.
template <int K, bool ADD2>
__global__ void __launch_bounds__(kRowThreads) combine_kernel(
    int64_t T, int vec_per_row, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ inv_pos, const uint4* __restrict__ Ys, const uint4* __restrict__ Ysh,
    const uint4* __restrict__ Ysh2, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t wglobal = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // kCombineSplit warps share a token row, each summing one contiguous part of it
  for (int64_t wt = wglobal; wt < T * kCombineSplit; wt += nwarps) {
    const int64_t t = wt / kCombineSplit;
    const int part = (int)(wt % kCombineSplit);
    const int per = (vec_per_row + kCombineSplit - 1) / kCombineSplit;
    const int v_begin = part * per;
    const int v_end = min(vec_per_row, v_begin + per);
    // order the token's routes by expert id (distinct experts)
    int pos[K];
    int ex[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      ex[j] = topk_idx[t * K + j];
      pos[j] = inv_pos[t * K + j];
    }
#pragma unroll
    for (int a = 1; a < K; ++a) {
#pragma unroll
      for (int b = K - 1; b >= a; --b) {
        const bool sw = ex[b] < ex[b - 1];
        const int e0 = ex[b - 1], e1 = ex[b], p0 = pos[b - 1], p1 = pos[b];
        ex[b - 1] = sw ? e1 : e0;
        ex[b] = sw ? e0 : e1;
        pos[b - 1] = sw ? p1 : p0;
        pos[b] = sw ? p0 : p1;
      }
    }
    float mul[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      mul[j] = pos[j] >= 0 ? 1.0f : 0.0f;
      pos[j] = max(pos[j], 0);
    }
    for (int v = v_begin + lane; v < v_end; v += 32) {
      uint4 q[K + 1];
      q[0] = Ysh ? Ysh[t * vec_per_row + v] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < K; ++j) q[j + 1] = Ys[(int64_t)pos[j] * vec_per_row + v];
      uint4 q2 = make_uint4(0, 0, 0, 0);
      if constexpr (ADD2) q2 = Ysh2[t * vec_per_row + v];
      float acc[8];
      acc[0] = bf16_lo(q[0].x); acc[1] = bf16_hi(q[0].x); acc[2] = bf16_lo(q[0].y); acc[3] = bf16_hi(q[0].y);
      acc[4] = bf16_lo(q[0].z); acc[5] = bf16_hi(q[0].z); acc[6] = bf16_lo(q[0].w); acc[7] = bf16_hi(q[0].w);
      if constexpr (ADD2) {
        acc[0] += bf16_lo(q2.x); acc[1] += bf16_hi(q2.x); acc[2] += bf16_lo(q2.y); acc[3] += bf16_hi(q2.y);
        acc[4] += bf16_lo(q2.z); acc[5] += bf16_hi(q2.z); acc[6] += bf16_lo(q2.w); acc[7] += bf16_hi(q2.w);
      }
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const uint4 u = q[j + 1];
        const float m = mul[j];
        acc[0] += m * bf16_lo(u.x); acc[1] += m * bf16_hi(u.x);
        acc[2] += m * bf16_lo(u.y); acc[3] += m * bf16_hi(u.y);
        acc[4] += m * bf16_lo(u.z); acc[5] += m * bf16_hi(u.z);
        acc[6] += m * bf16_lo(u.w); acc[7] += m * bf16_hi(u.w);
      }
      y[t * vec_per_row + v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

cudaError_t launch_combine(int64_t T, int d, int k, const int32_t* topk_idx, const int32_t* inv_pos,
                           const void* Ys, const void* Ysh, void* y, cudaStream_t s,
                           const void* Ysh2) {
  if (T == 0) return cudaSuccess;
  const auto ys = static_cast<const uint4*>(Ys);
  const auto ysh = static_cast<const uint4*>(Ysh);
  const auto ysh2 = static_cast<const uint4*>(Ysh2);
  auto yo = static_cast<uint4*>(y);
  const int grid = rows_grid(T * kCombineSplit);
  prof_begin("combine", s);
  auto launch = [&](auto kk) {
    constexpr int K = decltype(kk)::value;
    if (ysh2)
      combine_kernel<K, true><<<grid, kRowThreads, 0, s>>>(T, d / 8, topk_idx, inv_pos, ys, ysh, ysh2, yo);
    else
      combine_kernel<K, false><<<grid, kRowThreads, 0, s>>>(T, d / 8, topk_idx, inv_pos, ys, ysh, ysh2, yo);
  };
  switch (k) {
    case 1: launch(std::integral_constant<int, 1>{}); break;
    case 2: launch(std::integral_constant<int, 2>{}); break;
    case 3: launch(std::integral_constant<int, 3>{}); break;
    case 4: launch(std::integral_constant<int, 4>{}); break;
    case 5: launch(std::integral_constant<int, 5>{}); break;
    case 6: launch(std::integral_constant<int, 6>{}); break;
    case 7: launch(std::integral_constant<int, 7>{}); break;
    default: launch(std::integral_constant<int, 8>{}); break;
  }
  prof_end(s);
  return cudaGetLastError();
}

// Router backward for one token per warp.  dw_j = <dY_t, y_{e_j}(x_t)> is the fixed-order sum
// of the per-N-tile partials <a, h> written by the down-projection backward epilogue; with
// w_j = exp(l_j) / sum_{i in S} exp(l_i) (the renormalised softmax over the selection S),
// dl_m = w_m (dw_m - sum_j w_j dw_j) for m in S and 0 elsewhere.  Writes dlogits[T,E] fp32 and
// a bf16 copy dl[T,ldl] (columns E..ldl zero) that feeds the tensor-core GEMMs dl W_r^T, x^T dl.
__global__ void __launch_bounds__(kRowThreads) router_backward_kernel(
    int64_t T, int E, int k, int ldp, int ldl, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, const int32_t* __restrict__ inv_pos,
    const float* __restrict__ partial, float* __restrict__ dlogits, __nv_bfloat16* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int64_t wglobal = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = wglobal; t < T; t += nwarps) {
    float dw = 0.0f, w = 0.0f;
    int e = -1;
    if (lane < k) {
      const int64_t r = t * k + lane;
      e = topk_idx[r];
      w = topk_w[r];
      const int pos = inv_pos[r];
      if (pos >= 0)
        for (int n = 0; n < ldp; ++n) dw += partial[(int64_t)pos * ldp + n];
    }
    float inner = 0.0f;  // sum_j w_j dw_j in slot order, identical on every lane
    for (int j = 0; j < k; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const float dj = __shfl_sync(0xffffffffu, dw, j);
      inner += wj * dj;
    }
    const float dlj = w * (dw - inner);
    for (int c = lane; c < ldl; c += 32) {
      float v = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, e, j);
        const float vj = __shfl_sync(0xffffffffu, dlj, j);
        if (ej == c) v = vj;
      }
      if (c < E) dlogits[t * E + c] = v;
      dl[t * ldl + c] = __float2bfloat16_rn(v);
    }
  }
}

cudaError_t launch_router_backward(int64_t T, int E, int k, int ldp, const int32_t* topk_idx,
                                   const float* topk_w, const int32_t* inv_pos,
                                   const float* partial, float* dlogits, void* dl_bf16,
                                   cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int ldl = (E + 63) & ~63;
  prof_begin("router_bwd", s);
  router_backward_kernel<<<rows_grid(T), kRowThreads, 0, s>>>(
      T, E, k, ldp, ldl, topk_idx, topk_w, inv_pos, partial, dlogits,
      static_cast<__nv_bfloat16*>(dl_bf16));
  prof_end(s);
  return cudaGetLastError();
}

}  // namespace mok
