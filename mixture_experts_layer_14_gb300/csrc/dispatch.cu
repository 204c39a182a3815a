// Pull schedule of the MoE layer as a deterministic counting sort (page "Mixture-of-Kittens:
// Nhân kernel MoE ...", section "Lập lịch": scan the routing tensor and append every route to
// its expert's region, giving per-expert counts, region offsets and the schedule table; page
// "Метод и эксперименты": each expert then pulls its own tokens, e.g. E2 <- [0,2,9,15]).
//
// Four launches, no atomics on global memory, no host synchronisation:
//  1. histogram: block b counts, for every expert, the routes of tokens [64b, 64b+64) (one
//     thread per route; warp-level match gives per-warp counts);
//  2. scan: one block per expert turns its row of the (expert, block) histogram into exclusive
//     bases within the expert (in place) and its count;
//  3. offsets: one block scans the counts into region offsets;
//  4. scatter: block b gives route i of expert e the row offset(e) + base(e, b) + (routes of e in
//     earlier warps of the block) + (routes of e in lower lanes of its warp), i.e. routes keep
//     their (token, slot) order inside every region, so tokens ascend.
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

// Per expert (one block each, coalesced along its row of the histogram): the exclusive prefix of
// its per-chunk route counts, in place, and its total.
__global__ void __launch_bounds__(256) dispatch_scan_rows_kernel(int32_t* __restrict__ hist,
                                                                 int nblk,
                                                                 int32_t* __restrict__ counts) {
  __shared__ int s_warp[8];
  __shared__ int s_carry;
  int32_t* row = hist + (int64_t)blockIdx.x * nblk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < nblk; c0 += 256) {
    const int c = c0 + threadIdx.x;
    const int v = c < nblk ? row[c] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int below = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int x = s_warp[w];
      below += w < warp ? x : 0;
      total += x;
    }
    const int carry = s_carry;
    if (c < nblk) row[c] = carry + below + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry = carry + total;
    __syncthreads();
  }
  if (threadIdx.x == 0) counts[blockIdx.x] = s_carry;
}

// offsets[e] = routes of the experts before e, offsets[E] = all routes (one block, E <= 512).
__global__ void __launch_bounds__(kMaxE) dispatch_offsets_kernel(const int32_t* __restrict__ counts,
                                                                 int E,
                                                                 int32_t* __restrict__ offsets) {
  __shared__ int s_warp[kMaxE / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int v = t < E ? counts[t] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int below = 0;
  for (int w = 0; w < warp; ++w) below += s_warp[w];
  if (t < E) offsets[t] = below + incl - v;
  if (t == E - 1) offsets[E] = below + incl;
}

__global__ void __launch_bounds__(kDispatchChunk * kMaxK) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w, int64_t T, int E, int k,
    int nblk, const int32_t* __restrict__ offsets, const int32_t* __restrict__ base,
    int32_t* __restrict__ sorted_tok,
    float* __restrict__ sorted_w, int32_t* __restrict__ inv_pos) {
  __shared__ int s_cnt[kMaxDispatchWarps * kMaxE];
  int e;
  const int rank = warp_expert_rank(idx, T, E, k, blockIdx.x, s_cnt, nullptr, e);
  // exclusive prefix over the warps of the block, per expert, on top of the chunk's base (the
  // expert's offset plus the routes of its earlier chunks)
  const int nw = blockDim.x >> 5;
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = offsets[x] + base[(int64_t)x * nblk + blockIdx.x];
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
  dispatch_scan_rows_kernel<<<E, 256, 0, s>>>(hist, nblk, counts);
  prof_end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin("dispatch_offsets", s);
  dispatch_offsets_kernel<<<1, kMaxE, 0, s>>>(counts, E, offsets);
  prof_end(s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches += (nblk > 0) ? 3 : 2;
  if (nblk > 0) {
    prof_begin("dispatch_scatter", s);
    dispatch_scatter_kernel<<<nblk, kDispatchChunk * k, 0, s>>>(topk_idx, topk_w, T, E, k, nblk,
                                                                offsets, hist, sorted_tok, sorted_w,
                                                                inv_pos);
    prof_end(s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace mok
