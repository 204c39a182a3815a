// Pull schedule of the MoE layer as a deterministic counting sort (page "Mixture-of-Kittens:
// Nhân kernel MoE ...", section "Lập lịch": scan the routing tensor and append every route to
// its expert's region, giving per-expert counts, region offsets and the schedule table; page
// "Метод и эксперименты": each expert then pulls its own tokens, e.g. E2 <- [0,2,9,15]).
//
// Three launches, no atomics on global memory, no host synchronisation:
//  1. histogram: block b counts, for every expert, the routes of tokens [64b, 64b+64) (one
//     thread per route; warp-level match gives per-warp counts);
//  2. scan: one block turns the (expert, block) histogram, expert-major, into exclusive bases
//     (in place), per-expert counts and region offsets;
//  3. scatter: block b gives route i of expert e the row base(e, b) + (routes of e in earlier
//     warps of the block) + (routes of e in lower lanes of its warp), i.e. routes keep their
//     (token, slot) order inside every region, so tokens ascend.
#include "mok_device.cuh"

namespace mok {

constexpr int kMaxDispatchWarps = kDispatchChunk * kMaxK / 32;  // one thread per route

// Per-warp expert counts of a chunk's routes: thread i holds route i of the chunk (routes in
// token-major order).  __match_any_sync groups the lanes of a warp that route to the same
// expert; the lowest such lane writes the group size to s_cnt[warp][e], and every lane gets its
// rank inside its group (the number of lower lanes with the same expert).  No atomics.
__device__ __forceinline__ int warp_expert_rank(const int32_t* idx, int64_t T, int E, int k, int b,
                                                int* s_cnt, int* status, int& e_out) {
  const int64_t t0 = (int64_t)b * kDispatchChunk;
  const int64_t rem = T - t0;
  const int ntok = (int)(rem < kDispatchChunk ? rem : kDispatchChunk);
  const int n = ntok * k;
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  for (int j = i; j < kMaxDispatchWarps * E; j += blockDim.x) s_cnt[j] = 0;
  __syncthreads();
  int e = -1;
  if (i < n) {
    e = idx[t0 * k + i];
    if (e < 0 || e >= E) {
      if (status) record_status(status, MOK_ERR_DEVICE_CHECK);
      e = -1;  // the route is dropped
    }
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) s_cnt[warp * E + e] = __popc(peers);
  __syncthreads();
  e_out = e;
  return rank;
}

__global__ void __launch_bounds__(kDispatchChunk * kMaxK) dispatch_hist_kernel(
    const int32_t* __restrict__ idx, int64_t T, int E, int k, int nblk, int32_t* __restrict__ hist,
    int* status) {
  __shared__ int s_cnt[kMaxDispatchWarps * kMaxE];
  int e;
  warp_expert_rank(idx, T, E, k, blockIdx.x, s_cnt, status, e);
  const int nw = blockDim.x >> 5;
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int c = 0;
    for (int w = 0; w < nw; ++w) c += s_cnt[w * E + x];
    hist[(int64_t)x * nblk + blockIdx.x] = c;
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

__global__ void __launch_bounds__(kDispatchChunk * kMaxK) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w, int64_t T, int E, int k,
    int nblk, const int32_t* __restrict__ base, int32_t* __restrict__ sorted_tok,
    float* __restrict__ sorted_w, int32_t* __restrict__ inv_pos) {
  __shared__ int s_cnt[kMaxDispatchWarps * kMaxE];
  int e;
  const int rank = warp_expert_rank(idx, T, E, k, blockIdx.x, s_cnt, nullptr, e);
  // exclusive prefix over the warps of the block, per expert, on top of the chunk's base
  const int nw = blockDim.x >> 5;
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = base[(int64_t)x * nblk + blockIdx.x];
    for (int w = 0; w < nw; ++w) {
      const int c = s_cnt[w * E + x];
      s_cnt[w * E + x] = run;
      run += c;
    }
  }
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kDispatchChunk;
  const int64_t rem = T - t0;
  const int n = (int)(rem < kDispatchChunk ? rem : kDispatchChunk) * k;
  const int i = threadIdx.x;
  if (i < n) {
    const int64_t r = t0 * k + i;
    if (e >= 0) {
      const int pos = s_cnt[(i >> 5) * E + e] + rank;
      sorted_tok[pos] = (int32_t)(r / k);
      sorted_w[pos] = topk_w[r];
      inv_pos[r] = pos;
    } else {
      inv_pos[r] = -1;
    }
  }
}

cudaError_t launch_dispatch(int64_t T, int E, int k, const int32_t* topk_idx, const float* topk_w,
                            int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                            float* sorted_w, int32_t* inv_pos, int32_t* hist, int* status,
                            cudaStream_t s, int* launches) {
  const int nblk = (int)((T + kDispatchChunk - 1) / kDispatchChunk);
  if (nblk > 0) {
    prof_begin("dispatch_hist", s);
    dispatch_hist_kernel<<<nblk, kDispatchChunk * k, 0, s>>>(topk_idx, T, E, k, nblk, hist, status);
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
    dispatch_scatter_kernel<<<nblk, kDispatchChunk * k, 0, s>>>(topk_idx, topk_w, T, E, k, nblk,
                                                                hist, sorted_tok, sorted_w, inv_pos);
    prof_end(s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace mok
