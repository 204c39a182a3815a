// MXFP8 block quantisation (the MXFP8 path of the layer; page "Mixture-of-Kittens; MoE
// megakernel", key points: BF16 and MXFP8).  Format: E4M3 values with one UE8M0 power-of-two
// scale per 32 contiguous elements along the reduction dimension; the scale of a block is 2^s
// with s the smallest integer such that amax <= 448 * 2^s (amax / 448 rounded up to a power of
// two), s in [-127, 127], an all-zero block takes s = -127.  Values are multiplied by 2^-s
// (exact) and converted with cvt.rn.satfinite (round to nearest even, saturate to +-448).
#include "mok_mx.cuh"

namespace mok {

// rows x K bf16 (row-major) -> codes [rows][K] and scale bytes, [rows][K/32] or (ATOMS, K a
// multiple of 128) scale atoms by 128-row tile.  One warp per row, one 32-element block per lane
// per iteration.
template <bool ATOMS>
__global__ void __launch_bounds__(256) mx_quantize_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                               int64_t rows, int K,
                                                               uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ sc) {
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nblk = K / 32;
  for (int64_t r = w; r < rows; r += nw) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + r * K);
    uint4* q4 = reinterpret_cast<uint4*>(q + r * K);
    for (int b = lane; b < nblk; b += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = s4[b * 4 + i];
        const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * i + 2 * j] = bf16_lo(x[j]);
          v[8 * i + 2 * j + 1] = bf16_hi(x[j]);
        }
      }
      uint32_t qq[8];
      const uint32_t sb = mx_block32(v, qq);
      q4[b * 2] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
      q4[b * 2 + 1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
      if (ATOMS)
        sc[sf_atom_word(r >> 7, b >> 2, nblk >> 2, (int)(r & 127)) + (b & 3)] = (uint8_t)sb;
      else
        sc[r * nblk + b] = (uint8_t)sb;
    }
  }
}

// Weights: src [n][K][N] bf16 (row-major, the layer's x @ W layout) -> codes [n][N][K] (K-major,
// the operand layout of the block-scaled MMA) and scale atoms of the [n][N][K/32] scales, by
// 128-row tile of each matrix (N and K multiples of 128).  One thread per (matrix, column, K
// block): 32 strided reads (coalesced across the warp), 32 contiguous bytes out.
__global__ void __launch_bounds__(256) mx_quantize_transpose_kernel(
    const __nv_bfloat16* __restrict__ src, int64_t nmat, int K, int N, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sc) {
  const int nblk = K / 32;
  const int64_t total = nmat * (int64_t)nblk * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int col = (int)(i % N);
    const int64_t rest = i / N;
    const int kb = (int)(rest % nblk);
    const int64_t m = rest / nblk;
    const __nv_bfloat16* s = src + (m * K + (int64_t)kb * 32) * N + col;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __bfloat162float(s[(int64_t)j * N]);
    uint32_t qq[8];
    const uint32_t sb = mx_block32(v, qq);
    uint4* d = reinterpret_cast<uint4*>(q + (m * N + col) * (int64_t)K + (int64_t)kb * 32);
    d[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
    d[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
    sc[sf_atom_word(m * (N / 128) + col / 128, kb >> 2, nblk >> 2, col & 127) + (kb & 3)] = (uint8_t)sb;
  }
}

cudaError_t launch_mx_quantize_rows(const void* src, int64_t rows, int K, void* q, void* sc,
                                    bool atoms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 8);
  prof_begin("mx_quantize", s);
  auto k = atoms ? mx_quantize_rows_kernel<true> : mx_quantize_rows_kernel<false>;
  k<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), rows, K,
                                static_cast<uint8_t*>(q), static_cast<uint8_t*>(sc));
  prof_end(s);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_transpose(const void* src, int64_t nmat, int K, int N, void* q,
                                         void* sc, cudaStream_t s) {
  const int64_t total = nmat * (int64_t)(K / 32) * N;
  if (total == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)num_sms() * 16);
  prof_begin("mx_quantize_weights", s);
  mx_quantize_transpose_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src),
                                                           nmat, K, N, static_cast<uint8_t*>(q),
                                                           static_cast<uint8_t*>(sc));
  prof_end(s);
  return cudaGetLastError();
}

// Token-axis quantiser of the MXFP8 weight gradients (K = an expert's tokens): row i of expert e
// (source row rows_idx[offsets[e] + i], or offsets[e] + i) is column 128 s_mt[e] + i of a
// transposed code matrix q[C][128 nkb], s_mt being the prefix over experts of ceil(rows / 128);
// columns up to the expert's next multiple of 128 are zeros, so every 128-column K block of the
// GEMM holds one expert's tokens.  Blocks of 32 tokens start at the expert's first token.
// Tiled through shared memory, one 128-token x 64-column tile at a time: coalesced 128-byte
// row reads (gathered by rows_idx; the next tile's are issued before this one is quantised),
// one thread per (column, 32-token block) for the scale and codes, coalesced 128-byte column
// writes of the codes, one 4-byte atom word per column.  Up to three operands with the same
// rows and width go in one launch.
constexpr int kTokTile = 128, kColTile = 64;

__global__ void __launch_bounds__(256, 4) mx_quantize_tokens_kernel(const __grid_constant__ TokQuantParams tp) {
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_mt[kMaxE + 1];
  __shared__ uint32_t tile[kTokTile][kColTile / 2 + 1];  // bf16 pairs; odd pitch: no conflicts
  __shared__ __align__(16) uint8_t codes[kColTile][kTokTile + 16];
  __shared__ __align__(4) uint8_t sbytes[kColTile][4];
  const int tid = threadIdx.x;
  int E = tp.E;
  if (tp.offsets == nullptr) {
    if (tid == 0) {
      s_off[0] = 0;
      s_off[1] = (int)tp.nsrc;
      s_mt[0] = 0;
      s_mt[1] = (int)((tp.nsrc + 127) / 128);
    }
    E = 1;
  } else if (tid < 32) {  // one warp: offsets and the 128-column block prefix
    const int lane = tid;
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) local += (tp.offsets[e + 1] - tp.offsets[e] + 127) / 128;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        s_off[e] = tp.offsets[e];
        s_mt[e] = run;
        run += (tp.offsets[e + 1] - tp.offsets[e] + 127) / 128;
      }
    }
    if (lane == 31) {
      s_off[E] = tp.offsets[E];
      s_mt[E] = incl;
    }
  }
  __syncthreads();
  const int C = tp.C;
  const int64_t ld = 128 * (int64_t)tp.nkb;
  const int ncolt = C / kColTile;
  const int nkt = min(s_mt[E], tp.nkb);  // 128-token K blocks in use
  const int ntiles = tp.nops * nkt * ncolt;  // below 2^31: checked by the launcher
  const int ch = tid & 7;
  // tile id -> operand, K block and first column (column tiles fastest: neighbouring blocks read
  // the same source rows)
  auto decode = [&](int id, int& op, int& kt, int& c0) {
    op = id / (nkt * ncolt);
    const int rest = id - op * nkt * ncolt;
    kt = rest / ncolt;
    c0 = (rest - kt * ncolt) * kColTile;
  };
  // the tile's global loads, 128 rows x 64 columns: 8 threads per row, 16 bytes each, rows
  // tid / 8 + 32 j; rows past the expert's tokens are zeros
  auto fetch = [&](int id, uint4 (&u)[kTokTile / 32]) {
    int op, kt, c0;
    decode(id, op, kt, c0);
    int lo = 0, hi = E;  // the expert of K block kt: largest e with s_mt[e] <= kt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_mt[mid] <= kt) lo = mid; else hi = mid;
    }
    const int li0 = (kt - s_mt[lo]) * kTokTile;
    const int me = s_off[lo + 1] - s_off[lo];
    const __nv_bfloat16* src = tp.src[op];
#pragma unroll
    for (int j = 0; j < kTokTile / 32; ++j) {
      const int li = li0 + (tid >> 3) + 32 * j;
      u[j] = make_uint4(0u, 0u, 0u, 0u);
      if (li < me) {
        const int64_t row = s_off[lo] + li;
        const int64_t sr = tp.rows_idx ? (int64_t)tp.rows_idx[row] : row;
        if (sr >= 0 && sr < tp.nsrc) u[j] = *reinterpret_cast<const uint4*>(src + sr * C + c0 + 8 * ch);
      }
    }
  };
  uint4 u[kTokTile / 32];
  if ((int)blockIdx.x < ntiles) fetch(blockIdx.x, u);
  // two barriers per tile: the next tile's loads are in flight while this one is quantised
  for (int id = blockIdx.x; id < ntiles; id += gridDim.x) {
    int op, kt, c0;
    decode(id, op, kt, c0);
#pragma unroll
    for (int j = 0; j < kTokTile / 32; ++j) {
      const int r = (tid >> 3) + 32 * j;
      tile[r][4 * ch + 0] = u[j].x;
      tile[r][4 * ch + 1] = u[j].y;
      tile[r][4 * ch + 2] = u[j].z;
      tile[r][4 * ch + 3] = u[j].w;
    }
    __syncthreads();  // tile written; the previous tile's codes are out
    if (id + (int)gridDim.x < ntiles) fetch(id + gridDim.x, u);
    {  // thread: column cc, 32-token block b
      const int cc = tid & (kColTile - 1), b = tid >> 6;
      // the column's bf16 half of each word moved to the top 16 bits: one byte permute
      const uint32_t sel = (cc & 1) ? 0x3244u : 0x1044u;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(__byte_perm(tile[32 * b + i][cc >> 1], 0u, sel));
      uint32_t qq[8];
      sbytes[cc][b] = (uint8_t)mx_block32(v, qq);
      uint4* d = reinterpret_cast<uint4*>(&codes[cc][32 * b]);
      d[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
      d[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
    }
    __syncthreads();  // codes complete; the tile may be overwritten
    uint8_t* q = tp.q[op];
#pragma unroll
    for (int pass = 0; pass < kColTile / 32; ++pass) {  // 8 threads per column: 128 bytes
      const int cc = (tid >> 3) + 32 * pass;
      *reinterpret_cast<uint4*>(q + (int64_t)(c0 + cc) * ld + (int64_t)kt * kTokTile + 16 * ch) =
          *reinterpret_cast<const uint4*>(&codes[cc][16 * ch]);
    }
    if (tid < kColTile) {
      const int c = c0 + tid;
      *reinterpret_cast<uint32_t*>(tp.sc[op] + sf_atom_word(c >> 7, kt, tp.nkb, c & 127)) =
          *reinterpret_cast<const uint32_t*>(&sbytes[tid][0]);
    }
  }
}

cudaError_t launch_mx_quantize_tokens(const TokQuantParams& tp, cudaStream_t s) {
  const int64_t bound = (int64_t)tp.nops * tp.nkb * (tp.C / kColTile);  // tiles, upper bound
  if (bound == 0) return cudaSuccess;
  if (bound > 0x7fffffffLL) return cudaErrorInvalidValue;  // the kernel numbers tiles in an int
  // persistent: as many blocks as are resident at once, a property of this kernel on this device
  static int per_sm_of_device[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int per_sm = per_sm_of_device[dev];
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mx_quantize_tokens_kernel, 256, 0) !=
            cudaSuccess ||
        per_sm <= 0)
      per_sm = 4;
    per_sm_of_device[dev] = per_sm;
  }
  const int64_t blocks = std::min<int64_t>(bound, (int64_t)num_sms() * std::max(per_sm, 1));
  prof_begin("mx_quantize_tokens", s);
  mx_quantize_tokens_kernel<<<(int)blocks, 256, 0, s>>>(tp);
  prof_end(s);
  return cudaGetLastError();
}

// Scale atoms of the pulled rows: sorted row i (expert e, i - offsets[e] = 128 m + r) takes the
// scales of token sorted_tok[i] (atoms of x by 128-token tile) into row r of M tile s_mt[e] + m,
// s_mt being the prefix over experts of ceil(rows / 128), the M-grouped GEMM's tile order.  One
// 4-byte word (the row's four scales of one K block) per thread and (row, K block).
__global__ void __launch_bounds__(256) gather_scale_atoms_kernel(
    const uint8_t* __restrict__ src, const int32_t* __restrict__ sorted_tok,
    const int32_t* __restrict__ offsets, int E, int64_t T, int nkb, uint8_t* __restrict__ dst) {
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_mt[kMaxE + 1];
  if (threadIdx.x < 32) {  // one warp: offsets and the M-tile prefix
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) local += (offsets[e + 1] - offsets[e] + 127) / 128;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        s_off[e] = offsets[e];
        s_mt[e] = run;
        run += (offsets[e + 1] - offsets[e] + 127) / 128;
      }
    }
    if (lane == 31) s_off[E] = offsets[E];
  }
  __syncthreads();
  const int64_t R = s_off[E];
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < R * nkb;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int kb = (int)(i / R);
    const int row = (int)(i - (int64_t)kb * R);
    int lo = 0, hi = E;  // the expert holding sorted row `row`: largest e with s_off[e] <= row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= row) lo = mid; else hi = mid;
    }
    const int local = row - s_off[lo];
    const int64_t tok = sorted_tok[row];
    uint32_t w = 0u;
    if (tok >= 0 && tok < T)
      w = *reinterpret_cast<const uint32_t*>(src + sf_atom_word(tok >> 7, kb, nkb, (int)(tok & 127)));
    *reinterpret_cast<uint32_t*>(dst + sf_atom_word(s_mt[lo] + local / 128, kb, nkb, local & 127)) = w;
  }
}

cudaError_t launch_gather_scale_atoms(const void* src, const int32_t* sorted_tok,
                                      const int32_t* offsets, int E, int64_t T, int64_t R, int K,
                                      void* dst, cudaStream_t s) {
  if (R == 0 || E == 0) return cudaSuccess;
  const int nkb = K / 128;
  const int64_t blocks = std::min<int64_t>((R * nkb + 255) / 256, (int64_t)num_sms() * 8);
  prof_begin("gather_scale_atoms", s);
  gather_scale_atoms_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const uint8_t*>(src), sorted_tok,
                                                        offsets, E, T, nkb, static_cast<uint8_t*>(dst));
  prof_end(s);
  return cudaGetLastError();
}

}  // namespace mok
