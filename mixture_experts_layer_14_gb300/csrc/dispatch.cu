// Pull schedule of the MoE layer as a deterministic counting sort (page "Mixture-of-Kittens:
// Nhân kernel MoE ...", section "Lập lịch": scan the routing tensor and append every route to
// its expert's region, giving per-expert counts, region offsets and the schedule table; page
// "Метод и эксперименты": each expert then pulls its own tokens, e.g. E2 <- [0,2,9,15]).
//
// Three launches, no atomics on global memory, no host synchronisation:
//  1. histogram: block b counts, for every expert, the routes of tokens [64b, 64b+64);
//  2. scan: one block turns the (expert, block) histogram, expert-major, into exclusive bases
//     (in place), per-expert counts and region offsets;
//  3. scatter: block b walks its routes in (token, slot) order and gives each route of expert
//     e the next row of e's region, so tokens ascend inside every region.
#include "mok_device.cuh"

namespace mok {

constexpr int kDispatchThreads = 256;

__device__ __forceinline__ int load_chunk(const int32_t* idx, int64_t T, int E, int k, int b,
                                          int* s_idx, int* status) {
  const int64_t t0 = (int64_t)b * kDispatchChunk;
  const int64_t rem = T - t0;
  const int ntok = (int)(rem < kDispatchChunk ? rem : kDispatchChunk);
  const int n = ntok * k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int e = idx[t0 * k + i];
    if (e < 0 || e >= E) {
      record_status(status, MOK_ERR_DEVICE_CHECK);
      e = -1;  // the route is dropped
    }
    s_idx[i] = e;
  }
  __syncthreads();
  return n;
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_hist_kernel(
    const int32_t* __restrict__ idx, int64_t T, int E, int k, int nblk, int32_t* __restrict__ hist,
    int* status) {
  __shared__ int s_idx[kDispatchChunk * kMaxK];
  const int b = blockIdx.x;
  const int n = load_chunk(idx, T, E, k, b, s_idx, status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int cnt = 0;
    for (int i = 0; i < n; ++i) cnt += (s_idx[i] == e);
    hist[(int64_t)e * nblk + b] = cnt;
  }
}

__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int32_t* __restrict__ hist, int E,
                                                             int nblk, int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets) {
  __shared__ int s_warp[32];
  const int N = E * nblk;
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int i0 = threadIdx.x * per;
  const int i1 = min(N, i0 + per);
  int local = 0;
  for (int i = i0; i < i1; ++i) local += hist[i];
  // block-wide exclusive scan of the per-thread sums (thread order = entry order)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? s_warp[lane] : 0;
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += u;
    }
    if (lane < nw) s_warp[lane] = vi - v;  // exclusive warp base
  }
  __syncthreads();
  int run = s_warp[warp] + incl - local;
  for (int i = i0; i < i1; ++i) {
    const int h = hist[i];
    hist[i] = run;  // exclusive base of (expert, block), expert-major
    run += h;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int start = nblk ? hist[(int64_t)e * nblk] : 0;
    offsets[e] = start;
  }
  __syncthreads();
  if (threadIdx.x == blockDim.x - 1) offsets[E] = run;  // the last thread ends at the total
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = offsets[e + 1] - offsets[e];
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w, int64_t T, int E, int k,
    int nblk, const int32_t* __restrict__ base, int32_t* __restrict__ sorted_tok,
    float* __restrict__ sorted_w, int32_t* __restrict__ inv_pos, int* status) {
  __shared__ int s_idx[kDispatchChunk * kMaxK];
  const int b = blockIdx.x;
  const int n = load_chunk(idx, T, E, k, b, s_idx, nullptr);
  const int64_t r0 = (int64_t)b * kDispatchChunk * k;  // first route of the chunk
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int pos = base[(int64_t)e * nblk + b];
    for (int i = 0; i < n; ++i) {
      if (s_idx[i] == e) {
        const int64_t r = r0 + i;
        sorted_tok[pos] = (int32_t)(r / k);
        sorted_w[pos] = topk_w[r];
        inv_pos[r] = pos;
        ++pos;
      }
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (s_idx[i] < 0) inv_pos[r0 + i] = -1;
  (void)status;
}

cudaError_t launch_dispatch(int64_t T, int E, int k, const int32_t* topk_idx, const float* topk_w,
                            int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                            float* sorted_w, int32_t* inv_pos, int32_t* hist, int* status,
                            cudaStream_t s, int* launches) {
  const int nblk = (int)((T + kDispatchChunk - 1) / kDispatchChunk);
  if (nblk > 0) {
    prof_begin("dispatch_hist", s);
    dispatch_hist_kernel<<<nblk, kDispatchThreads, 0, s>>>(topk_idx, T, E, k, nblk, hist, status);
    prof_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  prof_begin("dispatch_scan", s);
  dispatch_scan_kernel<<<1, 1024, 0, s>>>(hist, E, nblk, counts, offsets);
  prof_end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches += (nblk > 0) ? 2 : 1;
  if (nblk > 0) {
    prof_begin("dispatch_scatter", s);
    dispatch_scatter_kernel<<<nblk, kDispatchThreads, 0, s>>>(topk_idx, topk_w, T, E, k, nblk, hist,
                                                              sorted_tok, sorted_w, inv_pos, status);
    prof_end(s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace mok
