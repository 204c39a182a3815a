// Router of the MoE layer: logits = x W_router + b on the tensor cores (tcgen05, fp32 TMEM
// accumulator), fused with the top-k selection and the renormalised softmax weights.  Page
// "Mixture-of-Kittens: Nhân kernel MoE ...", section "Chồng lấp tính toán và truyền tải trong
// MoE": the router projection picks the top-k routed experts of each token and gives each a
// router weight.
//
// One CTA per (128-token tile, K split).  Warp 0 issues TMA loads of the x tile (K-major) and of
// all E columns of W_router (MN-major), warp 1 issues the UMMAs (N = E rounded up to 64, split
// into MMAs of at most 256 columns), warps 2..9 run the epilogue, two per TMEM lane quarter.
// The bias is staged in shared memory once, so the epilogue reads it as broadcast vectors.
//  - One split (the token tiles alone fill the GPU): the two threads of a token row each select
//    the top k of half its columns straight from TMEM (loading the next 32 columns while they
//    rank the current ones), and the lower half inserts the upper half's list into its own
//    through shared memory.
//  - S > 1 splits (a power of two): the S CTAs of a tile form a thread-block cluster, and CTA r
//    reduces tile rows r 128/S .. (r+1) 128/S - 1.  Each CTA stores the partial logits of those
//    rows straight into CTA r's shared memory (the drained stage buffers, one slot per source
//    CTA, a chunk of columns at a time), so no thread waits on a remote load.  Then 2S threads
//    per row each sum the S partials of their share of the columns in rank order (the same
//    fixed order on every run), keep their own top-k list, and merge the lists with warp
//    shuffles.  The partial logits never leave the chip.
#include "mok_device.cuh"

namespace mok {

// Inserts (v, e) into the descending list (tv, ti): v lands before the first entry it strictly
// exceeds and the tail shifts down one place; nothing changes if it exceeds none (also for NaN).
// Experts arrive in ascending index order, so among equal logits the lower index stays ahead.
// Every slot's new value is computed from the old list alone, so the update is a few dependent
// instructions deep instead of a chain through all k slots.
__device__ __forceinline__ void topk_insert(float (&tv)[kMaxK], int (&ti)[kMaxK], float v, int e) {
  bool keep[kMaxK];  // slot j keeps its entry (v does not exceed it)
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) keep[j] = !(v > tv[j]);
#pragma unroll
  for (int j = kMaxK - 1; j >= 1; --j) {
    const bool here = !keep[j] && keep[j - 1];
    tv[j] = keep[j] ? tv[j] : (here ? v : tv[j - 1]);
    ti[j] = keep[j] ? ti[j] : (here ? e : ti[j - 1]);
  }
  tv[0] = keep[0] ? tv[0] : v;
  ti[0] = keep[0] ? ti[0] : e;
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

// (v, i) ranks before (bv, bi): larger logit first, lower expert index among equal logits; an
// empty entry (index -1) ranks last.
__device__ __forceinline__ bool ranks_before(float v, int i, float bv, int bi) {
  const unsigned ui = static_cast<unsigned>(i), ubi = static_cast<unsigned>(bi);
  return v > bv || (v == bv && ui < ubi);
}

// Merge of the sorted top-k lists of the S lanes of a group (lanes S g .. S g + S - 1) into the
// first k entries of (ov, oi), identical in every lane of the group.
template <int S>
__device__ __forceinline__ void merge_topk(int k, float (&tv)[kMaxK], int (&ti)[kMaxK],
                                           float (&ov)[kMaxK], int (&oi)[kMaxK]) {
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    ov[j] = -INFINITY;
    oi[j] = -1;
    if (j < k) {
      float bv = tv[0];
      int bi = ti[0];
#pragma unroll
      for (int o = 1; o < S; o <<= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, bv, o, S);
        const int i = __shfl_xor_sync(0xffffffffu, bi, o, S);
        if (ranks_before(v, i, bv, bi)) { bv = v; bi = i; }
      }
      // expert indices are distinct, so exactly one lane of the group holds the winner
      const bool mine = (bi == ti[0]) && (bi >= 0);
#pragma unroll
      for (int i = 0; i + 1 < kMaxK; ++i) {
        tv[i] = mine ? tv[i + 1] : tv[i];
        ti[i] = mine ? ti[i + 1] : ti[i];
      }
      if (mine) { tv[kMaxK - 1] = -INFINITY; ti[kMaxK - 1] = -1; }
      ov[j] = bv;
      oi[j] = bi;
    }
  }
}

// Splits > 1, one pass over logit columns c0 .. c0 + p.chunk - 1, after every CTA of the cluster
// has stored its partials of this CTA's rows: slot r of `part` holds CTA r's partial logits of
// rows rank 128/S .. (rank+1) 128/S - 1.  Epilogue thread `et` (0..255; 2S threads per row) sums
// the S partials of its row's columns 4 (sub + 2S i) .. + 3 in rank order, adds the bias and
// inserts them into its top-k list.
template <int S>
__device__ __forceinline__ void reduce_rows(const RouteParams& p, uint32_t part, uint32_t pstride,
                                            int c0, int rank, int et, const float* s_bias,
                                            float (&tv)[kMaxK], int (&ti)[kMaxK]) {
  constexpr int RPC = BM / S;           // rows this CTA reduces
  constexpr int TPR = 2 * S;            // threads per row
  const int row = et / TPR;             // of this CTA's rows
  const int sub = et % TPR;
  const int t = blockIdx.x * BM + rank * RPC + row;
  const uint32_t mine = part + row * pstride;
  const int n4 = p.chunk / 4;
  // two float4 columns per pass, every load issued first
  for (int j0 = sub; j0 < n4; j0 += 2 * TPR) {
    float4 v[2][S];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < S; ++r)
        v[h][r] = (j0 + h * TPR < n4) ? ld_shared_v4(mine + r * RPC * pstride + 16 * (j0 + h * TPR))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = j0 + h * TPR;
      if (j >= n4) break;
      float4 acc = v[h][0];
#pragma unroll
      for (int r = 1; r < S; ++r) {
        acc.x += v[h][r].x; acc.y += v[h][r].y; acc.z += v[h][r].z; acc.w += v[h][r].w;
      }
      const float4 b4 = reinterpret_cast<const float4*>(s_bias + c0)[j];
      const float a4[4] = {acc.x + b4.x, acc.y + b4.y, acc.z + b4.z, acc.w + b4.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = c0 + 4 * j + c;
        if (e < p.E) {
          if (t < p.T && p.logits) p.logits[(int64_t)t * p.E + e] = a4[c];
          topk_insert(tv, ti, a4[c], e);
        }
      }
    }
  }
}

template <int S>
__device__ __forceinline__ void finish_split(const RouteParams& p, int rank, int et,
                                             float (&tv)[kMaxK], int (&ti)[kMaxK]) {
  float ov[kMaxK];
  int oi[kMaxK];
  merge_topk<2 * S>(p.k, tv, ti, ov, oi);
  const int row = rank * (BM / S) + et / (2 * S);
  const int t = blockIdx.x * BM + row;
  if (et % (2 * S) == 0 && t < p.T) write_route(p, t, ov, oi);
}

constexpr int kRouteAuxBytes = 1024;  // barriers, TMEM address, abort flag
// warp 0 loads, warp 1 issues the MMAs, warps 2-9 run the epilogue: two per TMEM lane quarter
constexpr int kRouteThreads = 64 + 32 * 8;

__global__ void __launch_bounds__(kRouteThreads, 1) route_kernel(const __grid_constant__ RouteParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int E_pad = (p.E + 63) & ~63;
  const int a_bytes = BM * BK * 2;
  const int b_bytes = E_pad * BK * 2;
  const int stage_bytes = a_bytes + b_bytes;
  const int stages = min(4, (196608 / stage_bytes));
  const uint32_t pstride = 4u * p.chunk + 16u;  // a row of the partial-logit chunk
  const uint32_t region = max((uint32_t)(stages * stage_bytes), p.splits > 1 ? BM * pstride : 0u);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + stages * a_bytes;
  const uint32_t aux_s = base + region;
  uint8_t* aux = gbase + region;
  const uint32_t bar_full = aux_s;
  const uint32_t bar_empty = aux_s + 64;
  const uint32_t bar_acc = aux_s + 128;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(aux + 136);
  volatile int* s_abort = reinterpret_cast<volatile int*>(aux + 140);
  float* s_bias = reinterpret_cast<float*>(aux + kRouteAuxBytes);  // E_pad floats, zero past E
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
  for (int i = tid; i < E_pad; i += blockDim.x) s_bias[i] = (i < p.E && p.bias) ? p.bias[i] : 0.0f;
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  // top-k list of this thread (split path: of its row's columns)
  float tv[kMaxK];
  int ti[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) { tv[j] = -INFINITY; ti[j] = -1; }
  bool acc_ok = false;

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
    const int half = (warp - 2) >> 2;  // which of the two warps of this lane quarter
    const int r = q * 32 + lane;
    const int t = m0 + r;
    // the same in every lane: the warp's TMEM loads below need all 32 lanes
    acc_ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, 0, p.status, s_abort) ? 1 : 0) != 0;
    tc_fence_after();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    if (p.splits == 1) {
      // each of the two threads of a row ranks half of its 32-column chunks, loading the next 32
      // columns while it ranks the current ones (two named buffers, so both stay in registers)
      auto rank_cols = [&](const uint32_t (&v)[32], int c) {
        float b[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 b4 = reinterpret_cast<const float4*>(s_bias + c)[i];
          b[4 * i] = b4.x; b[4 * i + 1] = b4.y; b[4 * i + 2] = b4.z; b[4 * i + 3] = b4.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          if (e < p.E) {
            const float l = __uint_as_float(v[i]) + b[i];
            if (t < p.T && p.logits) p.logits[(int64_t)t * p.E + e] = l;
            topk_insert(tv, ti, l, e);
          }
        }
      };
      const int nch = (p.E + 31) / 32;  // 32 nch <= E_pad: every column loaded is allocated
      const int nh = (nch + 1) / 2;
      const int ch0 = half * nh, ch1 = min(nch, ch0 + nh);
      if (acc_ok && ch0 < ch1) {
        uint32_t va[32], vb[32];
        tmem_ld32(tacc + 32 * ch0, va);
        tmem_ld_wait();
        for (int ch = ch0; ch < ch1; ch += 2) {
          if (ch + 1 < ch1) tmem_ld32(tacc + 32 * (ch + 1), vb);
          rank_cols(va, 32 * ch);
          tmem_ld_wait();
          if (ch + 1 == ch1) break;
          if (ch + 2 < ch1) tmem_ld32(tacc + 32 * (ch + 2), va);
          rank_cols(vb, 32 * (ch + 1));
          tmem_ld_wait();
        }
      }
      // the upper half's list goes through shared memory (the drained stage buffers: every MMA
      // completed) to the lower half, which inserts it into its own: the lower half holds the
      // lower expert indices, so among equal logits its entries stay ahead
      uint32_t* lists = reinterpret_cast<uint32_t*>(gbase) + r * 16;
      if (half == 1) {
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
          lists[j] = __float_as_uint(tv[j]);
          lists[8 + j] = static_cast<uint32_t>(ti[j]);
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * 8) : "memory");  // the eight epilogue warps
      if (half == 0) {
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
          topk_insert(tv, ti, __uint_as_float(lists[j]), static_cast<int>(lists[8 + j]));
        if (acc_ok && t < p.T) write_route(p, t, tv, ti);
      }
    }
  }

  __syncwarp();  // the producer and MMA lanes rejoin their warps before any aligned barrier
  if (p.splits > 1) {
    // Every thread of every CTA of the cluster takes part in every cluster barrier below,
    // whatever happened above (a bounded wait that ran out leaves zeros), so none can wait
    // forever on a CTA that left.
    const int rank = (int)cluster_ctarank();
    const int et = tid - 64;  // epilogue thread 0..255
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const int rpc = BM / p.splits;  // rows each CTA of the cluster reduces
    // the drained stage buffers: slot r (rows r rpc .. r rpc + rpc - 1 of `part`) receives CTA
    // r's partials of this CTA's rows
    const uint32_t part = base;
    for (int c0 = 0; c0 < E_pad; c0 += p.chunk) {
      // every CTA of the cluster is past its MMAs (or the previous pass's reads): its stage
      // buffers may be written
      cluster_sync();
      if (warp >= 2) {
        const int rr = q * 32 + lane;  // tile row of this thread's TMEM lane
        const uint32_t dst = mapa_shared(part + (rank * rpc + rr % rpc) * pstride, rr / rpc);
        for (int cc = half * (p.chunk / 2); cc < (half + 1) * (p.chunk / 2); cc += 32) {
          uint32_t v[32];
          if (acc_ok && nkb > 0) {
            tmem_ld32(tacc + c0 + cc, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_cluster_v4(dst + 4 * cc + 16 * i, v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                 v[4 * i + 3]);
        }
      }
      cluster_sync();  // every partial of this pass is in its owner's shared memory
      if (warp >= 2) {
        if (p.splits == 2) reduce_rows<2>(p, part, pstride, c0, rank, et, s_bias, tv, ti);
        else if (p.splits == 4) reduce_rows<4>(p, part, pstride, c0, rank, et, s_bias, tv, ti);
        else reduce_rows<8>(p, part, pstride, c0, rank, et, s_bias, tv, ti);
      }
    }
    // no cluster barrier at the end: after the last pass's second one no CTA touches another's
    // shared memory, so each may leave when its own rows are done
    if (warp >= 2) {
      if (p.splits == 2) finish_split<2>(p, rank, et, tv, ti);
      else if (p.splits == 4) finish_split<4>(p, rank, et, tv, ti);
      else finish_split<8>(p, rank, et, tv, ti);
    }
  }
  if (warp >= 2) tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// K splits: the largest power of two (at most 8, at most one per k-block) such that the token
// tiles times the splits still fit on the GPU at once (T=4096 -> 4 splits of 28 k-blocks at
// d=7168; T=64 -> 8; from 152 SMs' worth of token tiles on, 1).
int route_splits(int64_t T, int d) {
  const int64_t mt = (T + BM - 1) / BM;
  const int nkb = d / BK;
  int sp = 1;
  while (2 * sp <= kMaxRouteSplits && 2 * sp <= nkb && mt * 2 * sp <= num_sms()) sp *= 2;
  return sp;
}

// Columns reduced per pass: all of E rounded up to 64 if 128 rows of them fit in the stage
// buffers, else half.
static int route_chunk(int E_pad, int region) {
  int ch = E_pad;
  while (ch > 32 && BM * (4 * ch + 16) > region) ch /= 2;
  return ch;
}

cudaError_t launch_route(const RouteParams& p_in, cudaStream_t s) {
  RouteParams p = p_in;
  const int E_pad = (p.E + 63) & ~63;
  const int stage_bytes = BM * BK * 2 + E_pad * BK * 2;
  const int stages = std::min(4, 196608 / stage_bytes);
  int region = stages * stage_bytes;
  p.chunk = route_chunk(E_pad, region);
  if (p.splits > 1) {
    if (p.chunk % 32 || E_pad % p.chunk || (p.splits != 2 && p.splits != 4 && p.splits != 8))
      return cudaErrorInvalidValue;
    region = std::max(region, BM * (4 * p.chunk + 16));
  }
  const int smem = region + kRouteAuxBytes + 4 * kMaxE + 1024;  // + 1024: base alignment
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.splits > 1 ? 1 : 0;
  cfg.gridDim = dim3((p.T + BM - 1) / BM, p.splits);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  prof_begin("route", s);
  e = cudaLaunchKernelEx(&cfg, route_kernel, p);
  prof_end(s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mok
