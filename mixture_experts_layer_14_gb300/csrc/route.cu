// Router of the MoE layer: logits = x W_router + b on the tensor cores (tcgen05, fp32 TMEM
// accumulator), fused with the top-k selection and the renormalised softmax weights in the
// epilogue.  Page "Mixture-of-Kittens: Nhân kernel MoE ...", section "Chồng lấp tính toán và
// truyền tải trong MoE": the router projection picks the top-k routed experts of each token and
// gives each a router weight.
//
// One CTA per 128-token tile.  Warp 0 issues TMA loads of the x tile (K-major) and of all E
// columns of W_router (MN-major), warp 1 issues the UMMAs (N = E rounded up to 64, split into
// MMAs of at most 256 columns), warps 2..5 run the epilogue: each thread owns one token row of
// the accumulator, so top-k needs no cross-thread communication.
#include "mok_device.cuh"

namespace mok {

__device__ __forceinline__ void topk_insert(float (&tv)[kMaxK], int (&ti)[kMaxK], float v, int e) {
  // Bubble (v, e) into the descending list.  Experts arrive in ascending index order and the
  // comparison is strict, so among equal logits the lower index stays ahead.
  float cv = v;
  int ci = e;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    const bool sw = cv > tv[j];
    const float ov = tv[j];
    const int oi = ti[j];
    tv[j] = sw ? cv : ov;
    ti[j] = sw ? ci : oi;
    cv = sw ? ov : cv;
    ci = sw ? oi : ci;
  }
}

// w_j = softmax(l)[e_j] / sum_sel softmax(l)[e_i] = exp(l_j - l_0) / sum_i exp(l_i - l_0)
__device__ __forceinline__ void write_route(const RouteParams& p, int t, const float (&tv)[kMaxK],
                                            const int (&ti)[kMaxK]) {
  float ex[kMaxK];
  float den = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    ex[j] = (j < p.k) ? __expf(tv[j] - tv[0]) : 0.0f;
    den += ex[j];
  }
  const float inv = 1.0f / den;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < p.k) {
      int e = ti[j];
      if (e < 0) {  // only possible with NaN logits
        record_status(p.status, MOK_ERR_DEVICE_CHECK);
        e = 0;
      }
      p.topk_idx[(int64_t)t * p.k + j] = e;
      p.topk_w[(int64_t)t * p.k + j] = ex[j] * inv;
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) route_kernel(const __grid_constant__ RouteParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int E_pad = (p.E + 63) & ~63;
  const int a_bytes = BM * BK * 2;
  const int b_bytes = E_pad * BK * 2;
  const int stage_bytes = a_bytes + b_bytes;
  const int stages = min(4, (196608 / stage_bytes));
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + stages * a_bytes;
  const uint32_t aux_s = base + stages * stage_bytes;
  uint8_t* aux = gbase + stages * stage_bytes;
  const uint32_t bar_full = aux_s;
  const uint32_t bar_empty = aux_s + 64;
  const uint32_t bar_acc = aux_s + 128;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(aux + 136);
  volatile int* s_abort = reinterpret_cast<volatile int*>(aux + 140);
  const uint32_t tmem_cols = E_pad <= 64 ? 64 : E_pad <= 128 ? 128 : E_pad <= 256 ? 256 : 512;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * BM;
  const int nkb_all = p.d / BK;
  const int kps = (nkb_all + p.splits - 1) / p.splits;  // k-blocks of this split
  const int kb0 = blockIdx.y * kps;
  const int nkb = max(0, min(nkb_all, kb0 + kps) - kb0);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.status, s_abort)) break;
        const uint32_t bar = bar_full + 8 * stage;
        mbar_arrive_expect_tx(bar, stage_bytes);
        tma_load_2d(sA0 + stage * a_bytes, &p.map_x, bar, (kb0 + kb) * BK, m0);
        for (int i = 0; i < E_pad / 64; ++i)
          tma_load_2d(sB0 + stage * b_bytes + i * 8192, &p.map_w, bar, 64 * i, (kb0 + kb) * BK);
        if (++stage == stages) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(bar_full + 8 * stage, phase, p.status, s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = sA0 + stage * a_bytes, sB = sB0 + stage * b_bytes;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = make_sdesc(sA + k * 32, 16, 1024);
          for (int c0 = 0; c0 < E_pad; c0 += 256) {
            const int n = min(256, E_pad - c0);
            const uint64_t bd = make_sdesc(sB + (c0 / 64) * 8192 + k * 2048, 8192, 1024);
            umma_bf16(tmem_base + c0, ad, bd, make_idesc_bf16(n, false, true), (kb | k) != 0);
          }
        }
        umma_commit(bar_empty + 8 * stage);
        if (++stage == stages) { stage = 0; phase ^= 1; }
      }
      umma_commit(bar_acc);  // also drains every MMA before TMEM is released
      if (!ok) {
        volatile int no_abort = 0;
        mbar_wait(bar_acc, 0, p.status, &no_abort);
      }
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int t = m0 + r;
    const bool ok = mbar_wait(bar_acc, 0, p.status, s_abort);
    tc_fence_after();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    if (ok && p.splits == 1) {
      float tv[kMaxK];
      int ti[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) { tv[j] = -INFINITY; ti[j] = -1; }
      for (int c = 0; c < p.E; c += 32) {
        uint32_t v[32];
        tmem_ld32(tacc + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          if (e < p.E) {
            const float l = __uint_as_float(v[i]) + (p.bias ? p.bias[e] : 0.0f);
            if (t < p.T && p.logits) p.logits[(int64_t)t * p.E + e] = l;
            if (l > tv[kMaxK - 1]) topk_insert(tv, ti, l, e);
          }
        }
      }
      if (t < p.T) write_route(p, t, tv, ti);
    } else if (ok) {
      // split K: store this split's partial logits; route_finish_kernel sums the splits
      float* part = p.partial + ((int64_t)blockIdx.y * p.T + t) * p.E;
      for (int c = 0; c < p.E; c += 32) {
        uint32_t v[32];
        tmem_ld32(tacc + c, v);
        tmem_ld_wait();
        if (t < p.T) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            if (c + i < p.E)
              *reinterpret_cast<float4*>(part + c + i) =
                  make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                              __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// Split-K router finish, one warp per token: sums the splits' partial logits in split order
// (bit-identical from run to run), adds the bias, then selects the top k with k rounds of a
// warp-shuffle argmax (larger logit first, lower expert index on ties) and writes the
// renormalised softmax weights.  Lane l holds experts l, l+32, ...; loads are coalesced.

// PER: logits per lane (E <= 32 PER), a compile-time size so that the arrays stay in registers
template <int PER>
__global__ void __launch_bounds__(256) route_finish_kernel(const __grid_constant__ RouteParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int per = (p.E + 31) / 32;
  for (int64_t t = w; t < p.T; t += nw) {
    float v[PER];
    bool used[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      used[i] = true;
      v[i] = -INFINITY;
      if (i < per && e < p.E) {
        // every split's partial in flight at once, then summed in split order
        float part[kMaxRouteSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxRouteSplits; ++sp)
          part[sp] = sp < p.splits ? __ldcg(p.partial + ((int64_t)sp * p.T + t) * p.E + e) : 0.0f;
        float acc = part[0];
#pragma unroll
        for (int sp = 1; sp < kMaxRouteSplits; ++sp)
          if (sp < p.splits) acc += part[sp];
        v[i] = acc + (p.bias ? p.bias[e] : 0.0f);
        used[i] = false;
        if (p.logits) p.logits[t * p.E + e] = v[i];
      }
    }
    float tv[kMaxK];
    int ti[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      tv[j] = -INFINITY;
      ti[j] = -1;
      if (j < p.k) {
        float best = -INFINITY;
        int bidx = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int e = lane + 32 * i;
          if (!used[i] && (v[i] > best || (v[i] == best && e < bidx))) { best = v[i]; bidx = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ob = __shfl_xor_sync(0xffffffffu, best, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
          if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
        }
        if (bidx != 0x7fffffff && (bidx & 31) == lane) {
#pragma unroll
          for (int i = 0; i < PER; ++i)
            if (i == (bidx >> 5)) used[i] = true;
        }
        tv[j] = best;
        ti[j] = (bidx == 0x7fffffff) ? -1 : bidx;
      }
    }
    if (lane == 0) write_route(p, (int)t, tv, ti);
  }
}

// K splits so that the grid fills the GPU about once (T=4096 -> 4 splits of 28 k-blocks at
// d=7168), at most route_splits_bound(); every split gets at least one k-block.
int route_splits(int64_t T, int d) {
  const int64_t mt = (T + BM - 1) / BM;
  const int nkb = d / BK;
  int sp = (int)std::max<int64_t>(1, num_sms() / std::max<int64_t>(mt, 1));
  sp = std::min(sp, route_splits_bound(T, d));
  const int kps = (nkb + sp - 1) / sp;
  return (nkb + kps - 1) / kps;
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t s) {
  const int E_pad = (p.E + 63) & ~63;
  const int stage_bytes = BM * BK * 2 + E_pad * BK * 2;
  const int stages = std::min(4, 196608 / stage_bytes);
  const int smem = stages * stage_bytes + 1024 + 1024;
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.T + BM - 1) / BM, p.splits);
  prof_begin("route", s);
  route_kernel<<<grid, kGemmThreads, smem, s>>>(p);
  prof_end(s);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t blocks = std::min<int64_t>((p.T + 7) / 8, (int64_t)num_sms() * 8);
  prof_begin("route_finish", s);
  const int per = (p.E + 31) / 32;
  if (per <= 2) route_finish_kernel<2><<<(int)blocks, 256, 0, s>>>(p);
  else if (per <= 4) route_finish_kernel<4><<<(int)blocks, 256, 0, s>>>(p);
  else if (per <= 8) route_finish_kernel<8><<<(int)blocks, 256, 0, s>>>(p);
  else route_finish_kernel<kMaxE / 32><<<(int)blocks, 256, 0, s>>>(p);
  prof_end(s);
  return cudaGetLastError();
}

}  // namespace mok
