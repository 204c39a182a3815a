// Persistent, warp-specialised grouped GEMM for the expert FFNs of the MoE layer (forward and
// backward), written for sm_103a with TMA, tcgen05.mma and TMEM accumulators.
//
// One CTA per SM.  Warp 0: TMA producer (one elected lane).  Warp 1: TMEM owner and UMMA
// issuer (one elected lane).  Warps 2..5: epilogue, one TMEM lane quarter each (thread = one
// output row).  A ring of STAGES shared-memory stages (A tile 128x64, B tile BNx64, both bf16
// in the 128-byte swizzled layout written by TMA) feeds the MMAs; two TMEM accumulators of BN
// fp32 columns let the epilogue of tile i overlap the MMAs of tile i+1.
//
// Scheduling: tiles are numbered on the device from the routing (pull schedule of the page
// "Mixture-of-Kittens: Nhân kernel MoE ...", section "Lập lịch": each expert's rows are a
// contiguous region of the destination buffer, so an expert's M tiles are contiguous row
// blocks pulled straight from it).  CTA c takes tiles c, c+grid, c+2*grid, ...  Every output
// element is produced by exactly one CTA with a fixed K order, so results are bit-identical
// from run to run.  No host synchronisation: the tile count is read on the device.
#include <algorithm>

#include "mok_nv.cuh"

namespace mok {

struct Tile {
  int g;     // 0 shared expert, 1 routed experts, 2 router GEMM (G_BWD_DW only)
  int e;     // expert index (coordinate of 3D weight maps; 0 for the shared expert)
  int sub;   // G_BWD_DW: 0 dW_gate, 1 dW_up, 2 dW_down
  int row0;  // M-grouped: first A row; K-grouped: first K row
  int rows;  // M-grouped: valid rows of the tile; K-grouped: K rows of the problem
  int m0;    // K-grouped: first output row (element offset along M)
  int n;     // N tile index
  int nkb;   // k-blocks
  int mt;    // M-grouped: index of the M tile in the decode order (shared tiles, then each
             // expert's); MXFP8 A scale atoms are stored by it
};

template <int MODE, int BN>
struct Cfg {
  // every stage row is 128 bytes: 64 bf16 or 128 E4M3 elements of K
  static constexpr bool MX = (MODE == G_FWD_GU_MX || MODE == G_FWD_DOWN_MX || MODE == G_BWD_DA_MX ||
                              MODE == G_BWD_DX_MX || MODE == G_BWD_DW_MX);
  // NVFP4: f16 A tiles by TMA; B arrives as E2M1 codes and E4M3 scales (32 + 4 bytes per row
  // of a 64-element K block) and converter warps decode it into an f16 K-major tile
  static constexpr bool NV = (MODE == G_FWD_GU_NV || MODE == G_FWD_DOWN_NV);
  static constexpr int KE = MX ? 128 : BK;            // K elements per stage
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  // UE8M0 atoms of A and B (MXFP8); the raw NVFP4 B rows (NVFP4)
  static constexpr int SF_BYTES = MX ? (BM + BN) * 4 : NV ? BN * 36 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
  static constexpr int STAGES = NV ? 4 : (BN == 256) ? 4 : 6;
  // NVFP4: three rings instead of one: STAGES A tiles; RAW_STAGES raw B rows, deep because they
  // come from HBM and are small (a stage is 9 KB against 48 KB of decoded f16), so the weight
  // stream runs far ahead of the MMA; DEC_STAGES decoded B tiles, which live only from the
  // converters to the MMA
  static constexpr int RAW_STAGES = NV ? 8 : 0;
  static constexpr int DEC_STAGES = NV ? 2 : 0;
  static constexpr bool A_MN = (MODE == G_BWD_DW);
  static constexpr bool B_MN = (MODE == G_FWD_GU || MODE == G_FWD_DOWN || MODE == G_BWD_DW ||
                                MODE == G_FWD_GUD);
  // gate/up then down in one launch, tiles claimed from a device work counter
  static constexpr bool FUSED = (MODE == G_FWD_GUD);
  // MXFP8: TMEM also holds the scale factors (from column 256), so one 256-column accumulator
  // or two of 128 columns
  static constexpr int NUM_ACC = (MX && BN == 256) ? 1 : 2;
  // epilogue warps: two per TMEM lane quarter (each taking half the columns) where the single
  // accumulator leaves the epilogue exposed, one otherwise
  static constexpr int EPI_WARPS = NUM_ACC == 1 ? 8 : 4;
  static constexpr int CONV_WARPS = NV ? 8 : 0;       // NVFP4 B decoders, after the epilogue warps
  // NVFP4: one more warp issues the raw B loads, so they do not wait behind the A ring
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + CONV_WARPS + (NV ? 1 : 0));
  // plain row-major outputs go through shared memory one 32-column chunk (32 rows x 64 B) per
  // epilogue warp at a time and are written with coalesced row stores
  static constexpr bool ROW_STAGED = (MODE == G_FWD_DOWN || MODE == G_BWD_DX ||
                                      MODE == G_FWD_DOWN_MX || MODE == G_BWD_DW ||
                                      MODE == G_BWD_DX_MX || MODE == G_BWD_DW_MX ||
                                      MODE == G_FWD_GUD || MODE == G_FWD_DOWN_NV);
  // per epilogue warp: a 2 KB row-staging buffer, or (dA MXFP8) a 32 x 36-float transpose buffer
  static constexpr int STG_STRIDE = (MODE == G_BWD_DA_MX) ? 32 * 36 * 4 : 2048;
  static constexpr int STAGING_BYTES = (ROW_STAGED || MODE == G_BWD_DA_MX) ? EPI_WARPS * STG_STRIDE : 0;
  static constexpr int TMEM_COLS = MX ? 512 : 2 * BN;
  static constexpr int RING_BYTES =
      NV ? STAGES * A_BYTES + DEC_STAGES * B_BYTES + RAW_STAGES * SF_BYTES : STAGES * STAGE_BYTES;
  static constexpr int SF_TMEM_COL = 256;              // MXFP8: 16 columns per stage from here
  static constexpr uint32_t IDESC =
      MX ? make_idesc_mxf8(BN) : NV ? make_idesc_f16(BN) : make_idesc_bf16(BN, A_MN, B_MN);
  static constexpr bool K_GROUPED = (MODE == G_BWD_DW || MODE == G_BWD_DW_MX);
};

constexpr int kAuxBytes = 1024;                      // barriers, TMEM address, abort flag, tile ring
constexpr int kRing = 4;                             // G_FWD_GUD: claimed tiles in flight per CTA
constexpr int kSchedBytes = 2 * (kMaxE + 1) * 4;     // expert row offsets + M-tile prefix

// PAIR: CTA-pair tiles (two CTAs of a cluster, M = 256, tcgen05.mma.cta_group::2).  Each CTA
// stages its own 128 A rows and half of the B columns, so a stage holds half the B bytes and six
// stages fit.
template <int MODE, int BN, bool PAIR>
struct KCfg : Cfg<MODE, BN> {
  using Base = Cfg<MODE, BN>;
  static_assert(!PAIR || (!Base::MX && BN == 256), "pairs: bf16, N = 256");
  static_assert(!PAIR || !Base::FUSED, "the fused forward runs single CTAs");
  static constexpr int B_BYTES = PAIR ? Base::B_BYTES / 2 : Base::B_BYTES;
  static constexpr int STAGE_BYTES = Base::A_BYTES + B_BYTES + Base::SF_BYTES;
  static constexpr int STAGES = PAIR ? 6 : Base::STAGES;
  static constexpr int RING_BYTES = PAIR ? STAGES * STAGE_BYTES : Base::RING_BYTES;
  static constexpr int BMT = PAIR ? 2 * BM : BM;  // rows of an M tile (M-grouped)
  static constexpr uint32_t IDESC =
      PAIR ? make_idesc_bf16(BN, Base::A_MN, Base::B_MN, 256) : Base::IDESC;
};

template <int MODE, int BN, bool PAIR = false>
constexpr int smem_bytes_for() {
  using C = KCfg<MODE, BN, PAIR>;
  return C::RING_BYTES + C::STAGING_BYTES + kAuxBytes + kSchedBytes + 1024;
}

// ------------------------------------------------------------------ tile decode
// PAIR: `tile` is a pair tile of 256 rows; CTA `rank` of the pair takes rows 128 rank ..
// 128 rank + 127 of it (rows past the group's end: t.rows <= 0, nothing stored).
template <int MODE, int BN, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, const int* s_off,
                                            const int* s_mt, int tile, int rank) {
  constexpr int BMT = KCfg<MODE, BN, PAIR>::BMT;
  Tile t;
  t.sub = 0;
  t.m0 = 0;
  t.mt = 0;
  if constexpr (!Cfg<MODE, BN>::K_GROUPED) {
    const int mt0 = p.has_shared ? (p.T + BMT - 1) / BMT : 0;
    int nt0 = p.nt[0], nt1 = p.nt[1];
    if constexpr (Cfg<MODE, BN>::FUSED) {  // the down tiles follow every gate/up tile
      const int tiles_a = mt0 * nt0 + (p.E > 0 ? s_mt[p.E] * nt1 : 0);
      if (tile >= tiles_a) {
        tile -= tiles_a;
        nt0 = p.ntb[0];
        nt1 = p.ntb[1];
        t.sub = 1;
      }
    }
    const int tiles0 = mt0 * nt0;
    if (tile < tiles0) {
      // a group with many M tiles runs N tiles fastest (its weights stay in L2 while its rows
      // stream once); otherwise M tiles fastest (one pass over each weight slice)
      const bool nfast = p.nfast_mt > 0 && mt0 >= p.nfast_mt;
      const int n = nfast ? tile % nt0 : tile / mt0;
      const int m = nfast ? tile / nt0 : tile - n * mt0;
      t.g = 0;
      t.e = 0;
      t.row0 = m * BMT + rank * BM;
      t.rows = min(BM, p.T - t.row0);
      t.n = n;
      t.mt = m;
    } else {
      const int l = tile - tiles0;
      const int nt = nt1;
      int lo = 0, hi = p.E;  // largest e with s_mt[e]*nt <= l
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_mt[mid] * nt <= l) lo = mid; else hi = mid;
      }
      const int e = lo;
      const int mte = s_mt[e + 1] - s_mt[e];
      const int l2 = l - s_mt[e] * nt;
      const bool nfast = p.nfast_mt > 0 && mte >= p.nfast_mt;
      const int n = nfast ? l2 % nt : l2 / mte;
      const int m = nfast ? l2 / nt : l2 - n * mte;
      t.g = 1;
      t.e = e;
      t.row0 = s_off[e] + m * BMT + rank * BM;
      t.rows = min(BM, s_off[e + 1] - t.row0);
      t.n = n;
      t.mt = s_mt[e] + m;
    }
    int nkb;
    if constexpr (MODE == G_FWD_GUD) nkb = t.sub ? (t.g ? p.F : p.Fs) / BK : p.d / BK;
    else if constexpr (MODE == G_FWD_GU || MODE == G_BWD_DA) nkb = p.d / BK;
    else if constexpr (MODE == G_FWD_DOWN) nkb = (t.g ? p.F : p.Fs) / BK;
    else if constexpr (MODE == G_FWD_GU_MX) nkb = p.d / 128;
    else if constexpr (MODE == G_FWD_DOWN_MX) nkb = (t.g ? p.F : p.Fs) / 128;
    else if constexpr (MODE == G_BWD_DA_MX) nkb = p.d / 128;
    else if constexpr (MODE == G_BWD_DX_MX) nkb = 2 * (t.g ? p.F : p.Fs) / 128;  // dG, then dU
    else if constexpr (MODE == G_FWD_GU_NV) nkb = p.d / BK;
    else if constexpr (MODE == G_FWD_DOWN_NV) nkb = (t.g ? p.F : p.Fs) / BK;
    else nkb = p.segkb[t.g][0] + p.segkb[t.g][1] + p.segkb[t.g][2];
    t.nkb = nkb;
  } else {
    // Inside a problem the N tiles run fastest, so the tiles in flight together write whole
    // output rows.  Pairs: the two CTAs take adjacent M tiles of the same N tile (every
    // problem's M-tile count is even).
    // divisions by the launch's divisors through their precomputed reciprocals (one wide
    // multiply each instead of an integer-division sequence on the issuing threads)
    constexpr int U = PAIR ? 2 : 1;
    auto div = [](int n, uint64_t m) { return (int)(((uint64_t)(uint32_t)n * m) >> 32); };
    auto place = [&](int ls, int nt, uint64_t mnt) {  // ls: tile index inside the problem
      const int ps = ls / U;
      const int q = div(ps, mnt);
      t.n = ps - q * nt;
      t.m0 = (q * U + ls % U) * BM;
    };
    int l = PAIR ? 2 * tile + rank : tile;
    if (l < p.router_tiles) {
      t.g = 2;
      t.e = 0;
      place(l, p.router_nt, p.dm_ntr);
      t.row0 = 0;
      t.rows = p.T;
    } else {
      l -= p.router_tiles;
      const int tiles_sh =
          p.has_shared ? 2 * (p.d / BM) * (p.Fs / BN) + (p.Fs / BM) * (p.d / BN) : 0;
      int Fg;
      if (l < tiles_sh) {
        t.g = 0;
        t.e = 0;
        Fg = p.Fs;
        t.row0 = 0;
        t.rows = p.T;
      } else {
        l -= tiles_sh;
        const int per = 2 * (p.d / BM) * (p.F / BN) + (p.F / BM) * (p.d / BN);
        const int e = div(l, p.dm_per);
        l -= e * per;
        t.g = 1;
        t.e = e;
        Fg = p.F;
        t.row0 = s_off[e];
        t.rows = s_off[e + 1] - s_off[e];
      }
      const int tg = (p.d / BM) * (Fg / BN);
      if (l < 2 * tg) {
        t.sub = l >= tg ? 1 : 0;
        place(l - t.sub * tg, Fg / BN, p.dm_nt[t.g]);
      } else {
        t.sub = 2;
        place(l - 2 * tg, p.d / BN, p.dm_ntd);
      }
    }
    if constexpr (MODE == G_BWD_DW_MX) {
      // transposed operands quantised along tokens: expert e's tokens are columns from
      // 128 s_mt[e] on, zero-padded to whole 128-column K blocks
      if (t.g == 1) t.row0 = 128 * s_mt[t.e];
      t.nkb = (t.rows + 127) / 128;
    } else {
      t.nkb = (t.rows + BK - 1) / BK;
    }
  }
  return t;
}

template <int MODE, int BN, bool PAIR>
__device__ __forceinline__ int total_tiles(const GemmParams& p, const int* s_mt) {
  if constexpr (!Cfg<MODE, BN>::K_GROUPED) {
    constexpr int BMT = KCfg<MODE, BN, PAIR>::BMT;
    const int mt0 = p.has_shared ? (p.T + BMT - 1) / BMT : 0;
    const int mte = p.E > 0 ? s_mt[p.E] : 0;
    if constexpr (Cfg<MODE, BN>::FUSED)
      return mt0 * (p.nt[0] + p.ntb[0]) + mte * (p.nt[1] + p.ntb[1]);
    return mt0 * p.nt[0] + mte * p.nt[1];
  } else {
    const int tiles_sh =
        p.has_shared ? 2 * (p.d / BM) * (p.Fs / BN) + (p.Fs / BM) * (p.d / BN) : 0;
    const int per = 2 * (p.d / BM) * (p.F / BN) + (p.F / BM) * (p.d / BN);
    return (p.router_tiles + tiles_sh + p.E * per) / (PAIR ? 2 : 1);
  }
}

// ------------------------------------------------------------------ producer
// G_BWD_DW, G_BWD_DW_MX: map slots of a tile's operands (g = 2: the router's x and dl).
__device__ __forceinline__ void dw_slots(const Tile& t, int& ia, int& ib) {
  if (t.g == 2) { ia = MS_R_A; ib = MS_R_B; }
  else if (t.sub == 0) { ia = t.g ? MS_A3 : MS_A0; ib = t.g ? MS_B3 : MS_B0; }
  else if (t.sub == 1) { ia = t.g ? MS_A3 : MS_A0; ib = t.g ? MS_B4 : MS_B1; }
  else { ia = t.g ? MS_A4 : MS_A1; ib = t.g ? MS_B5 : MS_B2; }
}

// Map slots per mode (g = group):
//  G_FWD_GU   A: x / x_sorted (K-major)            B: gate, up weights (MN-major, 3D)
//  G_FWD_DOWN A: h_sh / h (K-major)                B: down weights (MN-major, 3D)
//  G_BWD_DA   A: dY / dY_sorted (K-major)          B: down weights (K-major view, 3D)
//  G_BWD_DX   A: segments dG, dU (, dl)            B: gate, up (, router) weights (K-major view)
//  G_BWD_DW   A: x / x_sorted, w*h (MN-major)      B: dG, dU, dY (MN-major); router x, dl
//  MXFP8 (E4M3 codes, both K-major): gate/up A x, B gate, up; down A h, B down; da A dY, B down
//  quantised along d; dx A dG, dU, B gate, up quantised along F; dw A x^T, (w h)^T, B dG^T,
//  dU^T, dY^T (transposed, quantised along tokens)
// PAIR: each CTA loads its A rows and its half of B (gate/up: the gate columns in the even CTA,
// the up columns in the odd one; down: columns 128 rank .. 128 rank + 127 of the N tile), all
// completing on the even CTA's barrier (`bar` is a cluster address).
template <int MODE, int BN, bool PAIR>
__device__ __forceinline__ void issue_loads(const GemmParams& p, const Tile& t, int kb, int rank,
                                            uint32_t sA, uint32_t sB, uint32_t bar) {
  static_assert(!PAIR || MODE == G_FWD_GU || MODE == G_FWD_DOWN, "pair loads: gate/up and down");
  const CUtensorMap* M = p.maps;
  if constexpr (MODE == G_FWD_GUD) {
    if (t.sub == 0) {  // gate/up: as G_FWD_GU
      tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
      const CUtensorMap* bg = &M[t.g ? MS_B3 : MS_B0];
      const CUtensorMap* bu = &M[t.g ? MS_B4 : MS_B1];
      const int c0 = t.n * 128;
      tma_load_3d(sB + 0 * 8192, bg, bar, c0, kb * BK, t.e);
      tma_load_3d(sB + 1 * 8192, bg, bar, c0 + 64, kb * BK, t.e);
      tma_load_3d(sB + 2 * 8192, bu, bar, c0, kb * BK, t.e);
      tma_load_3d(sB + 3 * 8192, bu, bar, c0 + 64, kb * BK, t.e);
    } else {  // down: as G_FWD_DOWN, A = h (slots A1 / A4), B = down weights (B2 / B5)
      tma_load_2d(sA, &M[t.g ? MS_A4 : MS_A1], bar, kb * BK, t.row0);
      const CUtensorMap* b = &M[t.g ? MS_B5 : MS_B2];
#pragma unroll
      for (int i = 0; i < BN / 64; ++i) tma_load_3d(sB + i * 8192, b, bar, t.n * BN + 64 * i, kb * BK, t.e);
    }
  } else if constexpr (PAIR && MODE == G_FWD_GU) {
    tma_load_2d_pair(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
    const CUtensorMap* b = rank ? &M[t.g ? MS_B4 : MS_B1] : &M[t.g ? MS_B3 : MS_B0];
    const int c0 = t.n * 128;
    tma_load_3d_pair(sB, b, bar, c0, kb * BK, t.e);
    tma_load_3d_pair(sB + 8192, b, bar, c0 + 64, kb * BK, t.e);
  } else if constexpr (PAIR && MODE == G_FWD_DOWN) {
    tma_load_2d_pair(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
    const CUtensorMap* b = &M[t.g ? MS_B3 : MS_B0];
    const int c0 = t.n * BN + 128 * rank;
    tma_load_3d_pair(sB, b, bar, c0, kb * BK, t.e);
    tma_load_3d_pair(sB + 8192, b, bar, c0 + 64, kb * BK, t.e);
  } else if constexpr (MODE == G_FWD_GU) {
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
    const CUtensorMap* bg = &M[t.g ? MS_B3 : MS_B0];
    const CUtensorMap* bu = &M[t.g ? MS_B4 : MS_B1];
    const int c0 = t.n * 128;
    tma_load_3d(sB + 0 * 8192, bg, bar, c0, kb * BK, t.e);
    tma_load_3d(sB + 1 * 8192, bg, bar, c0 + 64, kb * BK, t.e);
    tma_load_3d(sB + 2 * 8192, bu, bar, c0, kb * BK, t.e);
    tma_load_3d(sB + 3 * 8192, bu, bar, c0 + 64, kb * BK, t.e);
  } else if constexpr (MODE == G_FWD_DOWN) {
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
    const CUtensorMap* b = &M[t.g ? MS_B3 : MS_B0];
#pragma unroll
    for (int i = 0; i < BN / 64; ++i) tma_load_3d(sB + i * 8192, b, bar, t.n * BN + 64 * i, kb * BK, t.e);
  } else if constexpr (MODE == G_FWD_GU_MX) {
    // E4M3 operands, both K-major: A = x rows, B = 128 gate rows then 128 up rows
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * 128, t.row0);
    tma_load_3d(sB, &M[t.g ? MS_B3 : MS_B0], bar, kb * 128, t.n * 128, t.e);
    tma_load_3d(sB + 16384, &M[t.g ? MS_B4 : MS_B1], bar, kb * 128, t.n * 128, t.e);
  } else if constexpr (MODE == G_FWD_DOWN_MX) {
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * 128, t.row0);
    tma_load_3d(sB, &M[t.g ? MS_B3 : MS_B0], bar, kb * 128, t.n * BN, t.e);
  } else if constexpr (MODE == G_BWD_DA_MX) {
    // E4M3 dY rows (K = d) and 256 rows of W_down quantised along d
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * 128, t.row0);
    tma_load_3d(sB, &M[t.g ? MS_B3 : MS_B0], bar, kb * 128, t.n * BN, t.e);
  } else if constexpr (MODE == G_BWD_DX_MX) {
    // k-blocks 0 .. F/128 - 1: dG with W_gate; then dU with W_up (both quantised along F)
    const int nseg = (t.g ? p.F : p.Fs) / 128;
    const int seg = kb >= nseg ? 1 : 0, kk = kb - seg * nseg;
    tma_load_2d(sA, &M[(t.g ? MS_A3 : MS_A0) + seg], bar, kk * 128, t.row0);
    tma_load_3d(sB, &M[(t.g ? MS_B3 : MS_B0) + seg], bar, kk * 128, t.n * BN, t.e);
  } else if constexpr (MODE == G_BWD_DW_MX) {
    // transposed operands [rows][K columns]: A rows m0.., B rows n BN.., K columns from row0
    int ia, ib;
    dw_slots(t, ia, ib);
    const int kc = t.row0 + kb * 128;
    tma_load_2d(sA, &M[ia], bar, kc, t.m0);
    tma_load_2d(sB, &M[ib], bar, kc, t.n * BN);
  } else if constexpr (MODE == G_BWD_DA) {
    tma_load_2d(sA, &M[t.g ? MS_A3 : MS_A0], bar, kb * BK, t.row0);
    tma_load_3d(sB, &M[t.g ? MS_B3 : MS_B0], bar, kb * BK, t.n * BN, t.e);
  } else if constexpr (MODE == G_FWD_GU_NV || MODE == G_FWD_DOWN_NV) {
    // f16 A rows (x values / h values); B comes raw through load_nv_raw.  A tile of at most 32
    // rows loads only those through the 32-row-box maps: the MMA's other rows are left as they
    // were, and the epilogue stores no row past t.rows
    const bool small = t.rows <= kNvSmallRows;
    tma_load_2d(sA, &M[t.g ? (small ? MS_A4 : MS_A3) : (small ? MS_A1 : MS_A0)], bar, kb * BK, t.row0);
  } else if constexpr (MODE == G_BWD_DX) {
    int seg = 0, kk = kb;
    while (seg < 2 && kk >= p.segkb[t.g][seg]) { kk -= p.segkb[t.g][seg]; ++seg; }
    tma_load_2d(sA, &M[(t.g ? MS_A3 : MS_A0) + seg], bar, kk * BK, t.row0);
    tma_load_3d(sB, &M[(t.g ? MS_B3 : MS_B0) + seg], bar, kk * BK, t.n * BN, seg == 2 ? 0 : t.e);
  } else {
    static_assert(MODE == -1, "every mode has its loads (G_BWD_DW: issue_loads_dw)");
  }
}

// G_BWD_DW loads of one k-block: A = the tile's 128 M columns of the K-row-major operand (two
// 64-column boxes), B = its BN N columns; `krow` = the block's first K row in the maps.
// PAIR: B columns 128 rank .. 128 rank + 127 of the tile only, on the even CTA's barrier.
template <int BN, bool PAIR>
__device__ __forceinline__ void issue_loads_dw(const CUtensorMap* ma, const CUtensorMap* mb,
                                               const Tile& t, int krow, int rank, uint32_t sA,
                                               uint32_t sB, uint32_t bar) {
  if constexpr (PAIR) {
    tma_load_2d_pair(sA, ma, bar, t.m0, krow);
    tma_load_2d_pair(sA + 8192, ma, bar, t.m0 + 64, krow);
    const int c0 = t.n * BN + 128 * rank;
    tma_load_2d_pair(sB, mb, bar, c0, krow);
    tma_load_2d_pair(sB + 8192, mb, bar, c0 + 64, krow);
  } else {
    tma_load_2d(sA, ma, bar, t.m0, krow);
    tma_load_2d(sA + 8192, ma, bar, t.m0 + 64, krow);
#pragma unroll
    for (int i = 0; i < BN / 64; ++i) tma_load_2d(sB + i * 8192, mb, bar, t.n * BN + 64 * i, krow);
  }
}

// ------------------------------------------------------------------ epilogues
__device__ __forceinline__ void st_row64(void* dst, const uint32_t (&v)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
__device__ __forceinline__ void ld_row64(const void* src, uint32_t (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = s[i];
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
}

// The warp no longer needs the accumulator: one arrival per warp on the accumulator-empty barrier
// at cluster address `release` (this CTA's, or the even CTA's of a CTA pair).
__device__ __forceinline__ void acc_release(uint32_t release, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(release);
}

// Staged row stores shared by the epilogues with plain row-major bf16 outputs.  Per 32-column
// chunk each thread's row (64 B) goes into the warp's 2 KB staging buffer (16-byte chunk i of row
// r at i ^ ((r / 2) % 4): conflict-free on both sides), then the warp reads it back by rows and
// stores eight whole 64-byte row pieces per instruction, skipping rows at or past `nrows` and
// columns at or past `ncols` (both counted from `o`, the warp's first row and column).
__device__ __forceinline__ void rows_store_chunk(__nv_bfloat16* o, int64_t ld, int nrows, int ncols,
                                                 uint32_t stg, int lane, const uint32_t (&P)[16]) {
  const uint32_t mine = stg + lane * 64;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(mine + ((i ^ ((lane >> 1) & 3)) << 4)),
                 "r"(P[4 * i]), "r"(P[4 * i + 1]), "r"(P[4 * i + 2]), "r"(P[4 * i + 3])
                 : "memory");
  __syncwarp();
  const int ch = lane & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2);  // rows 8j..8j+7, four 16-byte chunks each
    uint32_t a, b, c, d;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(stg + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4)));
    if (r < nrows && 8 * ch < ncols) *reinterpret_cast<uint4*>(o + r * ld + 8 * ch) = make_uint4(a, b, c, d);
  }
  __syncwarp();
}

__device__ __forceinline__ void pack_scaled(const uint32_t (&v)[32], float s, uint32_t (&P)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    P[i] = pack_bf16x2(s * __uint_as_float(v[2 * i]), s * __uint_as_float(v[2 * i + 1]));
}

// One warp's NCH x 32 accumulator columns (its TMEM lane quarter, from column `tcol`) times `s`
// (per thread: its row's factor) to bf16 rows through rows_store_chunk; `zero` writes zeros
// without reading TMEM.  The warp arrives on `release` once it no longer needs the accumulator:
// with EARLY, after packing every column into registers (the next tile's MMAs then run under the
// stores); otherwise at the end, with the TMEM load of the next chunk in flight during each
// chunk's stores.
template <int NCH, bool EARLY>
__device__ __forceinline__ void store_acc_rows(__nv_bfloat16* o, int64_t ld, int nrows, int ncols,
                                               uint32_t tcol, bool zero, float s, uint32_t stg,
                                               int lane, uint32_t release) {
  if (nrows <= 0 || ncols <= 0) {
    acc_release(release, lane);
    return;
  }
  if constexpr (EARLY) {
    static_assert(NCH % 2 == 0, "pairs of chunks");
    uint32_t P[NCH][16];
#pragma unroll
    for (int c = 0; c < NCH; c += 2) {
      uint32_t v[2][32];
      if (!zero) {
        tmem_ld32(tcol + 32 * c, v[0]);
        tmem_ld32(tcol + 32 * c + 32, v[1]);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[0][i] = v[1][i] = 0u;
      }
      pack_scaled(v[0], s, P[c]);
      pack_scaled(v[1], s, P[c + 1]);
    }
    acc_release(release, lane);
#pragma unroll
    for (int c = 0; c < NCH; ++c)
      rows_store_chunk(o + 32 * c, ld, nrows, ncols - 32 * c, stg, lane, P[c]);
  } else {
    uint32_t v[2][32];
    if (!zero) tmem_ld32(tcol, v[0]);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      uint32_t P[16];
      if (!zero) {
        tmem_ld_wait();
        pack_scaled(v[c & 1], s, P);
        if (c + 1 < NCH) tmem_ld32(tcol + 32 * (c + 1), v[(c + 1) & 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) P[i] = 0u;
      }
      rows_store_chunk(o + 32 * c, ld, nrows, ncols - 32 * c, stg, lane, P);
    }
    acc_release(release, lane);
  }
}

// Columns of one epilogue warp: all BN with four epilogue warps, half with eight.
template <int MODE, int BN>
constexpr int warp_cols() { return Cfg<MODE, BN>::EPI_WARPS == 8 ? BN / 2 : BN; }

// G_FWD_DOWN, G_FWD_DOWN_MX (Y_s = router weight x accumulator; the shared expert's rows take
// weight 1), G_BWD_DX and G_BWD_DX_MX (dX_s = accumulator): row-major outputs with d columns,
// rows past the expert's last token skipped.
template <int MODE, int BN>
__device__ __forceinline__ void epilogue_rows(const GemmParams& p, void* const (&outs)[2], const Tile& t,
                                              uint32_t tacc, uint32_t stg, int q, int half, int lane,
                                              uint32_t release) {
  constexpr int cols = warp_cols<MODE, BN>();
  const int nrows = t.rows - q * 32;  // valid rows among this warp's 32 (may be <= 0)
  constexpr bool WEIGHTED = (MODE == G_FWD_DOWN || MODE == G_FWD_DOWN_MX || MODE == G_FWD_DOWN_NV);
  float s = 1.0f;
  if (WEIGHTED && t.g == 1 && lane < nrows) s = p.row_w[t.row0 + q * 32 + lane];
  // NVFP4: the two tensor scales, h's and the expert's down weight's
  if constexpr (MODE == G_FWD_DOWN_NV) s *= __fmul_rn(nv_decode_g(p.nv_act[1]), p.nvg[t.g][0][t.e]);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(outs[t.g]) + (int64_t)(t.row0 + q * 32) * p.d +
                     t.n * BN + cols * half;
  store_acc_rows<cols / 32, Cfg<MODE, BN>::NUM_ACC == 1>(o, p.d, nrows, cols, tacc + cols * half,
                                                         false, s, stg, lane, release);
}

// G_BWD_DW, G_BWD_DW_MX: weight gradients [d x F] (dW_gate, dW_up), [F x d] (dW_down) or
// [d x E] (router); an expert without tokens gets zeros.
template <int MODE, int BN>
__device__ __forceinline__ void epilogue_dw(const GemmParams& p, const Tile& t, uint32_t tacc,
                                            uint32_t stg, int q, int half, int lane,
                                            uint32_t release) {
  using bf16 = __nv_bfloat16;
  constexpr int cols = warp_cols<MODE, BN>();
  bf16* out;
  int ld, ncols;
  if (t.g == 2) {
    out = static_cast<bf16*>(p.out_router);
    ld = ncols = p.E_cols;
  } else {
    const int Fg = t.g ? p.F : p.Fs;
    if (t.sub < 2) {
      out = static_cast<bf16*>(t.sub ? p.out1[t.g] : p.out0[t.g]) + (int64_t)t.e * p.d * Fg;
      ld = Fg;
    } else {
      out = static_cast<bf16*>(p.out2[t.g]) + (int64_t)t.e * Fg * p.d;
      ld = p.d;
    }
    ncols = ld;
  }
  const int col0 = t.n * BN + cols * half;
  store_acc_rows<cols / 32, Cfg<MODE, BN>::NUM_ACC == 1>(out + (int64_t)(t.m0 + 32 * q) * ld + col0,
                                                         ld, 32, ncols - col0, tacc + cols * half,
                                                         t.nkb == 0, 1.0f, stg, lane, release);
}

// G_FWD_GU_MX: h = SiLU(g) * u quantised per 32 columns into E4M3 codes [rows][F] and UE8M0
// scale atoms by M tile; the tile's 128 h columns are K block t.n of the down projection.  This
// warp takes h columns 64*half .. 64*half+63 of the tile: both 32-column blocks are computed and
// quantised in registers, the accumulator is released (the next tile's MMAs then run under the
// stores), then the codes and scale bytes are written.  Training (out2 set): g and u are also
// stored in fp32 (out2, out3), as accumulated, for the backward's requantisation.
template <int BN>
__device__ __forceinline__ void epilogue_gu_mx(const GemmParams& p, const Tile& t, uint32_t tacc,
                                               int r, int half, uint32_t release) {
  uint32_t qq[2][8], sb[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int c = 64 * half + 32 * b;
    uint32_t gr[32], ur[32];
    tmem_ld32(tacc + c, gr);
    tmem_ld32(tacc + 128 + c, ur);
    tmem_ld_wait();
    float hv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) hv[i] = silu_f(__uint_as_float(gr[i])) * __uint_as_float(ur[i]);
    sb[b] = mx_block32(hv, qq[b]);
    if (p.out2[t.g] && r < t.rows) {
      const int64_t o = (int64_t)(t.row0 + r) * (t.g ? p.F : p.Fs) + t.n * 128 + c;
      uint4* gd = reinterpret_cast<uint4*>(static_cast<float*>(p.out2[t.g]) + o);
      uint4* ud = reinterpret_cast<uint4*>(static_cast<float*>(p.out3[t.g]) + o);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gd[i] = make_uint4(gr[4 * i], gr[4 * i + 1], gr[4 * i + 2], gr[4 * i + 3]);
        ud[i] = make_uint4(ur[4 * i], ur[4 * i + 1], ur[4 * i + 2], ur[4 * i + 3]);
      }
    }
  }
  acc_release(release, r & 31);
  if (r < t.rows) {
    const int ld = t.g ? p.F : p.Fs;
    uint8_t* hq = static_cast<uint8_t*>(p.out0[t.g]) + (int64_t)(t.row0 + r) * ld + t.n * 128 + 64 * half;
    uint4* d = reinterpret_cast<uint4*>(hq);
    d[0] = make_uint4(qq[0][0], qq[0][1], qq[0][2], qq[0][3]);
    d[1] = make_uint4(qq[0][4], qq[0][5], qq[0][6], qq[0][7]);
    d[2] = make_uint4(qq[1][0], qq[1][1], qq[1][2], qq[1][3]);
    d[3] = make_uint4(qq[1][4], qq[1][5], qq[1][6], qq[1][7]);
    // scale bytes of blocks 2*half and 2*half+1: adjacent bytes of the row's atom word
    uint8_t* hs = static_cast<uint8_t*>(p.out1[t.g]) + sf_atom_word(t.mt, t.n, ld / 128, r) + 2 * half;
    *reinterpret_cast<uint16_t*>(hs) = (uint16_t)(sb[0] | (sb[1] << 8));
  }
}

// Token-axis MXFP8 quantisation of one 32-column chunk held by a warp whose 32 lanes are 32
// consecutive tokens of one expert (one 32-token block): v[j] = the lane's value in column
// c0 + j.  The chunk is transposed through the warp's shared-memory buffer (element (column j,
// token i) at float 36 j + i: conflict-free writes, 16-byte reads), then lane j quantises column
// c0 + j's 32 tokens and stores their codes as 32 consecutive bytes of that column's row of the
// transposed matrix (`col0` points at column c0, token column of lane 0), and its scale byte as
// block q of K block kg.
__device__ __forceinline__ void quant_tokens_chunk(const float (&v)[32], uint32_t stg, uint8_t* col0,
                                                   int64_t ld, uint8_t* atoms, int c0, int kg,
                                                   int nkb, int q, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + 4u * (36u * j + lane)), "f"(v[j]) : "memory");
  __syncwarp();
  float col[32];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(col[4 * i]), "=f"(col[4 * i + 1]), "=f"(col[4 * i + 2]), "=f"(col[4 * i + 3])
                 : "r"(stg + 4u * (36u * lane + 4u * i)));
  __syncwarp();  // the buffer is rewritten by the next chunk
  uint32_t qq[8];
  const uint32_t sb = mx_block32(col, qq);
  uint4* d = reinterpret_cast<uint4*>(col0 + (int64_t)lane * ld);
  d[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
  d[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
  const int c = c0 + lane;
  atoms[sf_atom_word(c >> 7, kg, nkb, c & 127) + q] = (uint8_t)sb;
}

// G_BWD_DA_MX: from a = dY W_down^T (the accumulator) and the saved G, U (fp32): dG and dU
// quantised per 32 columns (E4M3 codes [rows][F] and scale atoms by M tile: the A operands of the
// block-scaled dX GEMM); dG, dU and w*h quantised along tokens (the warp's 32 rows are one
// 32-token block of one expert) into the transposed operands of the weight-gradient GEMM; and
// the router partial <a, h> per (routed row, 128-column block).  This warp takes columns
// 128 half .. 128 half + 127 of the tile (N tile 128 with two accumulators and four epilogue
// warps: half = 0): K block kb of F, whose four scale bytes per row are one atom word.  Rows past
// the expert's last token count as zeros in the token blocks.
__device__ __forceinline__ void ld_row128(const float* src, float (&v)[32]) {
  const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = s[i];
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
}

template <int BN>
__device__ __forceinline__ void epilogue_da_mx(const GemmParams& p, const Tile& t, uint32_t tacc,
                                               uint32_t stg, int q, int half, int lane,
                                               uint32_t release) {
  const int r = q * 32 + lane;
  const bool valid = r < t.rows;
  const int ld = t.g ? p.F : p.Fs;
  const int64_t row = t.row0 + r;
  const float w = (t.g == 1 && valid) ? p.row_w[row] : 1.0f;
  const int kb = t.n * (BN / 128) + half;
  const int64_t off = row * ld + 128 * kb;
  const float* Gs = static_cast<const float*>(p.in0[t.g]) + off;
  const float* Us = static_cast<const float*>(p.in1[t.g]) + off;
  uint8_t* dGq = static_cast<uint8_t*>(p.qout[t.g][0]) + off;
  uint8_t* dUq = static_cast<uint8_t*>(p.qout[t.g][1]) + off;
  const int nkbt = p.tnkb[t.g];
  const int64_t tld = 128 * (int64_t)nkbt;
  const int64_t kpos = 128 * (int64_t)t.mt + 32 * q;  // the warp's token columns
  float pacc = 0.0f;
  uint32_t sg = 0u, su = 0u;
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    float gq[32], uq[32];  // G and U of this chunk (their loads overlap the TMEM load)
    if (valid) {
      ld_row128(Gs + c, gq);
      ld_row128(Us + c, uq);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) gq[i] = uq[i] = 0.0f;
    }
    uint32_t v[32];
    tmem_ld32(tacc + 128 * half + c, v);
    tmem_ld_wait();
    const int col0 = 128 * kb + c;
    float f[32];
    uint32_t qq[8];
    // dG = w a u s (1 + g (1 - s)), s = sigmoid(g); gq then holds SiLU(g) = g s
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float g = gq[i], u = uq[i];
      const float sgm = sigmoid_f(g);
      f[i] = valid ? w * __uint_as_float(v[i]) * u * sgm * (1.0f + g * (1.0f - sgm)) : 0.0f;
      gq[i] = g * sgm;
    }
    if (valid) {
      sg |= mx_block32(f, qq) << (c / 4);  // scale byte c / 32 of the row's atom word
      uint4* dq = reinterpret_cast<uint4*>(dGq + c);
      dq[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
      dq[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
    }
    quant_tokens_chunk(f, stg, p.tq[t.g][0] + (int64_t)col0 * tld + kpos, tld, p.tsc[t.g][0], col0,
                       t.mt, nkbt, q, lane);
    // dU = w a SiLU(g)
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = valid ? w * __uint_as_float(v[i]) * gq[i] : 0.0f;
    if (valid) {
      su |= mx_block32(f, qq) << (c / 4);
      uint4* dq = reinterpret_cast<uint4*>(dUq + c);
      dq[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
      dq[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
    }
    quant_tokens_chunk(f, stg, p.tq[t.g][1] + (int64_t)col0 * tld + kpos, tld, p.tsc[t.g][1], col0,
                       t.mt, nkbt, q, lane);
    // w h, h = g s u, and the router partial <a, h>
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float hv = gq[i] * uq[i];
      pacc += __uint_as_float(v[i]) * hv;  // zero on rows past the expert (g = u = 0)
      f[i] = w * hv;
    }
    quant_tokens_chunk(f, stg, p.tq[t.g][2] + (int64_t)col0 * tld + kpos, tld, p.tsc[t.g][2], col0,
                       t.mt, nkbt, q, lane);
  }
  acc_release(release, lane);
  if (valid) {
    *reinterpret_cast<uint32_t*>(p.qsc[t.g][0] + sf_atom_word(t.mt, kb, ld / 128, r)) = sg;
    *reinterpret_cast<uint32_t*>(p.qsc[t.g][1] + sf_atom_word(t.mt, kb, ld / 128, r)) = su;
    if (t.g == 1) p.partial[row * (ld / 128) + kb] = pacc;
  }
}

// G_FWD_GU_NV: G and U are the accumulators times their tensor scales (x's and the expert's gate
// or up weight's); h = SiLU(G) * U is quantised per 16 columns with h's calibrated tensor amax and
// stored as f16 NVFP4 values without the tensor scale: the A operand of the NVFP4 down GEMM.
template <int BN>
__device__ __forceinline__ void epilogue_gu_nv(const GemmParams& p, const Tile& t, uint32_t tacc, int r) {
  const bool valid = r < t.rows;
  const int ld = t.g ? p.F : p.Fs;
  const float gx = nv_decode_g(p.nv_act[0]);
  const float ag = __fmul_rn(gx, p.nvg[t.g][0][t.e]);
  const float au = __fmul_rn(gx, p.nvg[t.g][1][t.e]);
  const float Sh = nv_tensor_S(p.nv_act[1]);
  __half* h = static_cast<__half*>(p.out0[t.g]) + (int64_t)(t.row0 + r) * ld + t.n * 128;
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    uint32_t gr[32], ur[32];
    tmem_ld32(tacc + c, gr);
    tmem_ld32(tacc + 128 + c, ur);
    tmem_ld_wait();
    if (valid) {
      float hv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        hv[i] = silu_f(ag * __uint_as_float(gr[i])) * (au * __uint_as_float(ur[i]));
      uint32_t o[16];
      nv_block16_values(hv, Sh, o);
      nv_block16_values(hv + 16, Sh, o + 8);
      st_row64(h + c, o);
    }
  }
}

template <int MODE, int BN>
__device__ __forceinline__ void epilogue(const GemmParams& p, const Tile& t, uint32_t tacc,
                                         int r, int half) {
  using bf16 = __nv_bfloat16;
  static_assert(MODE == G_FWD_GU || MODE == G_BWD_DA, "the other modes have their own epilogues");
  if constexpr (MODE == G_FWD_GU) {
    const bool valid = r < t.rows;
    const int ld = t.g ? p.F : p.Fs;
    const int64_t row = t.row0 + r;
    bf16* h = static_cast<bf16*>(p.out0[t.g]) + row * ld + t.n * 128;
    bf16* G = p.out1[t.g] ? static_cast<bf16*>(p.out1[t.g]) + row * ld + t.n * 128 : nullptr;
    bf16* U = p.out2[t.g] ? static_cast<bf16*>(p.out2[t.g]) + row * ld + t.n * 128 : nullptr;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t gr[32], ur[32];
      tmem_ld32(tacc + c, gr);
      tmem_ld32(tacc + 128 + c, ur);
      tmem_ld_wait();
      if (valid) {
        uint32_t hp[16], gp[16], up[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
          const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
          hp[i] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
          gp[i] = pack_bf16x2(g0, g1);
          up[i] = pack_bf16x2(u0, u1);
        }
        st_row64(h + c, hp);
        if (G) st_row64(G + c, gp);
        if (U) st_row64(U + c, up);
      }
    }
  } else if constexpr (MODE == G_BWD_DA) {
    const bool valid = r < t.rows;
    const int ld = t.g ? p.F : p.Fs;
    const int64_t row = t.row0 + r;
    const float w = (t.g == 1 && valid) ? p.row_w[row] : 1.0f;
    const int64_t off = row * ld + t.n * BN;
    const bf16* Gs = static_cast<const bf16*>(p.in0[t.g]) + off;
    const bf16* Us = static_cast<const bf16*>(p.in1[t.g]) + off;
    bf16* dG = static_cast<bf16*>(p.out0[t.g]) + off;
    bf16* dU = static_cast<bf16*>(p.out1[t.g]) + off;
    bf16* hw = static_cast<bf16*>(p.out2[t.g]) + off;
    float pacc = 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      tmem_ld32(tacc + c, v);
      tmem_ld_wait();
      if (valid) {
        uint32_t gq[16], uq[16], o0[16], o1[16], o2[16];
        ld_row64(Gs + c, gq);
        ld_row64(Us + c, uq);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float res[2][3];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float g = h2 ? bf16_hi(gq[i]) : bf16_lo(gq[i]);
            const float u = h2 ? bf16_hi(uq[i]) : bf16_lo(uq[i]);
            const float a = __uint_as_float(v[2 * i + h2]);
            const float sg = sigmoid_f(g);
            const float hv = g * sg * u;
            pacc += a * hv;
            const float dh = w * a;
            res[h2][0] = dh * u * sg * (1.0f + g * (1.0f - sg));
            res[h2][1] = dh * g * sg;
            res[h2][2] = w * hv;
          }
          o0[i] = pack_bf16x2(res[0][0], res[1][0]);
          o1[i] = pack_bf16x2(res[0][1], res[1][1]);
          o2[i] = pack_bf16x2(res[0][2], res[1][2]);
        }
        st_row64(dG + c, o0);
        st_row64(dU + c, o1);
        st_row64(hw + c, o2);
      }
    }
    if (valid && t.g == 1) p.partial[row * p.nt[1] + t.n] = pacc;
  }
}

// ------------------------------------------------------------------ MXFP8 scale factors
// Writes the stage's UE8M0 scale factors into shared memory in the layout tcgen05.cp
// (32x128b, replicated to the four lane quarters) moves into TMEM: a 512-byte atom per 128 rows
// in which row r = r0 + 32*r1 (r0 < 32, r1 < 4) keeps its four K-block scales (K elements
// kb*128 + 32*j, j = 0..3, byte j) at offset 16*r0 + 4*r1.  Scale rows are row-major [rows][K/32]
// in global memory, so the four bytes of a row are one aligned 32-bit word.
// MXFP8: the stage's scale atoms (the A tile's, then one per 128 B rows) by bulk copies on the
// stage barrier.  Gate/up: B rows 0-127 are gate rows, 128-255 up rows of the h tile; down, da,
// dx: B rows are 256 consecutive rows of the expert's K-major weight (two atoms); dw: A and B
// rows are rows of the transposed operands, K block t.row0 / 128 + kb of the whole matrix.
template <int MODE, int BN>
__device__ __forceinline__ void load_scale_atoms(const GemmParams& p, const Tile& t, int kb,
                                                 uint32_t sf, uint32_t bar) {
  const int nkb = p.sf_kb[t.g];
  if constexpr (MODE == G_FWD_GU_MX) {
    bulk_load(sf, p.sfa[t.g][0] + sf_atom_word(t.mt, kb, nkb, 0), 512, bar);
    const int64_t tile = (int64_t)t.e * p.nt[t.g] + t.n;  // 128-row tile of gate / up
    bulk_load(sf + 512, p.sfb[t.g][0] + sf_atom_word(tile, kb, nkb, 0), 512, bar);
    bulk_load(sf + 1024, p.sfb[t.g][1] + sf_atom_word(tile, kb, nkb, 0), 512, bar);
  } else if constexpr (MODE == G_FWD_DOWN_MX || MODE == G_BWD_DA_MX || MODE == G_BWD_DX_MX) {
    int seg = 0, kk = kb;
    if constexpr (MODE == G_BWD_DX_MX) {  // dG with gate, then dU with up: nkb blocks each
      seg = kb >= nkb ? 1 : 0;
      kk = kb - seg * nkb;
    }
    bulk_load(sf, p.sfa[t.g][seg] + sf_atom_word(t.mt, kk, nkb, 0), 512, bar);
    // the BN weight rows of the N tile: BN / 128 row tiles of the expert's K-major weight
    const int64_t tile = ((int64_t)t.e * p.nt[t.g] + t.n) * (BN / 128);
#pragma unroll
    for (int a = 0; a < BN / 128; ++a)
      bulk_load(sf + 512 * (1 + a), p.sfb[t.g][seg] + sf_atom_word(tile + a, kk, nkb, 0), 512, bar);
  } else if constexpr (MODE == G_BWD_DW_MX) {
    const int kg = t.row0 / 128 + kb;
    const uint8_t* a = p.sfa[t.g][t.sub == 2 ? 1 : 0];
    const uint8_t* b = p.sfb[t.g][t.sub];
    bulk_load(sf, a + sf_atom_word(t.m0 / 128, kg, nkb, 0), 512, bar);
    bulk_load(sf + 512, b + sf_atom_word(2 * t.n, kg, nkb, 0), 512, bar);
    bulk_load(sf + 1024, b + sf_atom_word(2 * t.n + 1, kg, nkb, 0), 512, bar);
  } else {
    static_assert(MODE == -1, "scale atoms of an MXFP8 mode");
  }
}

// ------------------------------------------------------------------ NVFP4 B operand
// The stage's raw B rows by bulk copies on the stage barrier: BN rows of 32 code bytes, then BN
// rows of 4 scale bytes.  Gate/up: rows 0-127 are the gate rows, 128-255 the up rows of the h
// tile's 128 columns; down: 256 consecutive rows (output columns) of the expert's weight.
template <int MODE, int BN>
__device__ __forceinline__ void load_nv_raw(const GemmParams& p, const Tile& t, int kb, uint32_t raw,
                                            uint32_t bar) {
  const int g = t.g;
  if constexpr (MODE == G_FWD_GU_NV) {
    const int N = g ? p.F : p.Fs;
    const int64_t row = ((int64_t)t.e * (p.d / BK) + kb) * N + t.n * 128;
    bulk_load(raw, p.nvq[g][0] + row * 32, 128 * 32, bar);
    bulk_load(raw + 128 * 32, p.nvq[g][1] + row * 32, 128 * 32, bar);
    bulk_load(raw + BN * 32, p.nvs[g][0] + row * 4, 128 * 4, bar);
    bulk_load(raw + BN * 32 + 128 * 4, p.nvs[g][1] + row * 4, 128 * 4, bar);
  } else if constexpr (MODE == G_FWD_DOWN_NV) {
    const int64_t row = ((int64_t)t.e * ((g ? p.F : p.Fs) / BK) + kb) * p.d + t.n * BN;
    bulk_load(raw, p.nvq[g][0] + row * 32, BN * 32, bar);
    bulk_load(raw + BN * 32, p.nvs[g][0] + row * 4, BN * 4, bar);
  } else {
    static_assert(MODE == -1, "raw B rows of an NVFP4 mode");
  }
}

// Converter thread `ct` (0..NCT-1) decodes B rows ct, ct + NCT, ... of a stage: each row's 64 codes
// times their block scales into f16, written K-major with the 128-byte swizzle the MMA reads
// (row n: 8-row group n / 8 at 1024 bytes, row n % 8 at 128 bytes, 16-byte chunk c at c ^ (n % 8)).
// Rows sit 32 bytes apart, so the eight lanes of one 16-byte load phase would meet in pairs on
// the same banks; lanes with bit 2 of the row set read their second half first instead.
template <int BN, int NCT>
__device__ __forceinline__ void nv_convert_stage(uint32_t raw, uint32_t sB, int ct) {
#pragma unroll 1
  for (int n = ct; n < BN; n += NCT) {
    uint32_t w[8], v[8];
    const uint32_t h = (n & 4) ? 16u : 0u;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(raw + n * 32 + h));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]) : "r"(raw + n * 32 + (16u - h)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = h ? v[i + 4] : v[i];
      w[i + 4] = h ? v[i] : v[i + 4];
    }
    uint32_t sc;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(raw + BN * 32 + n * 4));
    const uint32_t row = sB + (n >> 3) * 1024 + (n & 7) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // K elements 8c .. 8c + 7, scale block c / 2
      const uint32_t s2 = e4m3_bcast_f16x2((sc >> (8 * (c >> 1))) & 0xFFu);
      uint32_t o[4];
      e2m1x8_to_f16x2(w[c], o);
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = hmul2_u32(o[j], s2);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ (n & 7)) << 4)),
                   "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                   : "memory");
    }
  }
}

// ------------------------------------------------------------------ K-tail masking
// G_BWD_DW: the last k-block of a problem may hold rows of the next expert; zero them in both
// operands (MN-major: K is the row index inside every 64-column box, 128 B per row, and the
// 128-byte swizzle only permutes 16-byte chunks within a row).

// ------------------------------------------------------------------ the kernel
// PAIR: launched in clusters of two CTAs; the pair takes one 256-row tile at a time.  The even
// CTA issues the MMAs (cta_group::2) once both CTAs' stage has landed on its full barrier and
// multicasts its commits to the empty and accumulator-full barriers of both CTAs; every
// epilogue warp of both CTAs arrives on the even CTA's accumulator-empty barrier.
template <int MODE, int BN, bool PAIR>
__global__ void __launch_bounds__(Cfg<MODE, BN>::THREADS, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = KCfg<MODE, BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + C::STAGES * C::A_BYTES;
  // MXFP8 scale-factor atoms; NVFP4 raw B rows
  const uint32_t sSF0 = sB0 + (C::NV ? C::DEC_STAGES : C::STAGES) * C::B_BYTES;
  const uint32_t sSTG0 = base + C::RING_BYTES;  // output staging of the epilogue warps
  uint8_t* aux = gbase + C::RING_BYTES + C::STAGING_BYTES;
  const uint32_t aux_s = base + C::RING_BYTES + C::STAGING_BYTES;
  // aux layout: full[S] empty[S] tfull[2] tempty[2] drain | tmem addr | abort
  const uint32_t bar_full = aux_s;
  const uint32_t bar_empty = aux_s + 8 * C::STAGES;
  const uint32_t bar_tfull = aux_s + 16 * C::STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(aux + 16 * C::STAGES + 40);
  volatile int* s_abort = reinterpret_cast<volatile int*>(aux + 16 * C::STAGES + 48);
  // G_FWD_GUD: a ring of claimed tile indices (full: written by the producer; empty: taken by the
  // MMA warp and every epilogue warp)
  const uint32_t bar_rfull = aux_s + 16 * C::STAGES + 64;
  const uint32_t bar_rempty = bar_rfull + 8 * kRing;
  volatile int* s_ring = reinterpret_cast<volatile int*>(aux + 16 * C::STAGES + 64 + 16 * kRing);
  // NVFP4, in the tile ring's space (unused): decoded B tile full (one arrival per converter
  // warp) and empty (MMA commit), raw B rows full (bulk copies) and empty (converter warps)
  const uint32_t bar_conv = aux_s + 16 * C::STAGES + 64;
  const uint32_t bar_dempty = bar_conv + 8 * C::DEC_STAGES;
  const uint32_t bar_rawfull = bar_dempty + 8 * C::DEC_STAGES;
  const uint32_t bar_rawempty = bar_rawfull + 8 * C::RAW_STAGES;
  static_assert(16 * C::STAGES + 64 + 16 * (C::DEC_STAGES + C::RAW_STAGES) <= kAuxBytes, "aux barriers");
  int* s_off = reinterpret_cast<int*>(aux + kAuxBytes);
  int* s_mt = s_off + (kMaxE + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, C::EPI_WARPS * (PAIR ? 2 : 1));  // one arrival per warp
    }
    mbar_init(bar_drain, 1);
    if constexpr (C::FUSED) {
      for (int i = 0; i < kRing; ++i) {
        mbar_init(bar_rfull + 8 * i, 1);
        mbar_init(bar_rempty + 8 * i, 1 + C::EPI_WARPS);
      }
    }
    if constexpr (C::NV) {
      static_assert(!C::FUSED, "the decoded-B barriers use the tile ring's space");
      for (int s = 0; s < C::DEC_STAGES; ++s) {
        mbar_init(bar_conv + 8 * s, C::CONV_WARPS);
        mbar_init(bar_dempty + 8 * s, 1);
      }
      for (int s = 0; s < C::RAW_STAGES; ++s) {
        mbar_init(bar_rawfull + 8 * s, 1);
        mbar_init(bar_rawempty + 8 * s, C::CONV_WARPS);
      }
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < MS_COUNT; ++i) tma_prefetch_desc(&p.maps[i]);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(s_tmem), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(s_tmem), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == 2 && p.E > 0) {
    // expert row offsets and (M-grouped) the prefix of M tiles per expert, one warp
    const int per = (p.E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < p.E) {
        const int o0 = p.offsets[e], o1 = p.offsets[e + 1];
        s_off[e] = o0;
        local += (o1 - o0 + C::BMT - 1) / C::BMT;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < p.E) {
        s_mt[e] = run;
        run += (p.offsets[e + 1] - p.offsets[e] + C::BMT - 1) / C::BMT;
      }
    }
    if (lane == 31) {
      s_mt[p.E] = incl;
      s_off[p.E] = p.offsets[p.E];
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int ntiles = total_tiles<MODE, BN, PAIR>(p, s_mt);
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // tile loop of this CTA
  const int step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (warp == 0) {
    if constexpr (MODE == G_BWD_DW) {
      // A routed tile's K rows are one expert's rows: its loads go through that expert's copies
      // of the A and B maps, bounded to its rows (dw_bound_maps_kernel), so the rows past its end
      // arrive as zeros.  A map is acquired from the tensor-map proxy when it changes.
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        const CUtensorMap* last_a = nullptr;
        const CUtensorMap* last_b = nullptr;
        for (int tile = first; tile < ntiles && !*s_abort; tile += step) {
          const Tile t = decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank);
          if (t.nkb == 0) continue;
          int ia, ib;
          dw_slots(t, ia, ib);
          const CUtensorMap* ma = &p.maps[ia];
          const CUtensorMap* mb = &p.maps[ib];
          int krow = t.row0;
          if (t.g == 1) {
            ma = p.emaps + (size_t)t.e * kBoundMaps + (ia == MS_A3 ? 0 : 1);
            mb = p.emaps + (size_t)t.e * kBoundMaps + (ib - MS_B3 + 2);
            if (ma != last_a) tmap_acquire(ma);
            if (mb != last_b) tmap_acquire(mb);
            last_a = ma;
            last_b = mb;
            krow = 0;
          }
          bool ok = true;
          for (int kb = 0; kb < t.nkb; ++kb) {
            if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.status, s_abort)) { ok = false; break; }
            if (!PAIR || rank == 0)
              mbar_arrive_expect_tx(bar_full + 8 * stage, (C::A_BYTES + C::B_BYTES) * (PAIR ? 2 : 1));
            issue_loads_dw<BN, PAIR>(ma, mb, t, krow + kb * BK, rank, sA0 + stage * C::A_BYTES,
                                     sB0 + stage * C::B_BYTES,
                                     PAIR ? mapa_shared(bar_full + 8 * stage, 0) : bar_full + 8 * stage);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
        }
      }
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      auto produce = [&](const Tile& t) {
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.status, s_abort)) return;
          // a pair's stage: both CTAs' bytes on the even CTA's barrier; NVFP4: A only
          const uint32_t kTx = C::NV ? (t.rows <= kNvSmallRows ? kNvSmallRows * 128 : C::A_BYTES)
                                     : C::A_BYTES + C::B_BYTES + C::SF_BYTES;
          if (!PAIR || rank == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, kTx * (PAIR ? 2 : 1));
          issue_loads<MODE, BN, PAIR>(p, t, kb, rank, sA0 + stage * C::A_BYTES,
                                      sB0 + stage * C::B_BYTES,
                                      PAIR ? mapa_shared(bar_full + 8 * stage, 0) : bar_full + 8 * stage);
          if constexpr (C::MX)
            load_scale_atoms<MODE, BN>(p, t, kb, sSF0 + stage * C::SF_BYTES, bar_full + 8 * stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      };
      if constexpr (C::FUSED) {
        // claim tiles in order from the work counter and hand each to the MMA and epilogue warps;
        // a down tile first waits until every gate/up tile of its M tile has written its h rows
        const int mt0 = p.has_shared ? (p.T + BM - 1) / BM : 0;
        for (int it = 0;; ++it) {
          const int slot = it % kRing;
          if (!mbar_wait(bar_rempty + 8 * slot, ((it / kRing) & 1) ^ 1, p.status, s_abort)) break;
          const int tile = *s_abort ? ntiles : atomicAdd(p.work, 1);
          s_ring[slot] = tile;
          mbar_arrive(bar_rfull + 8 * slot);
          if (tile >= ntiles) break;
          const Tile t = decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank);
          if (t.sub == 1 && !wait_counter(p.ready + (t.g ? mt0 + t.mt : t.mt), p.nt[t.g] * C::EPI_WARPS,
                                          p.status, s_abort))
            break;
          produce(t);
        }
      } else {
        for (int tile = first; tile < ntiles && !*s_abort; tile += step)
          produce(decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank));
      }
    }
  } else if (warp == 1 && (!PAIR || rank == 0)) {
    int stage = 0;
    uint32_t phase = 0;
    int ds = 0;  // NVFP4: decoded B ring
    uint32_t dphase = 0;
    // the MMAs of the it-th tile of this CTA; false when a bounded wait ran out
    auto mma_tile = [&](const Tile& t, int it) -> bool {
      const int buf = it % C::NUM_ACC;
      const uint32_t tph = (it / C::NUM_ACC) & 1;
      if (!mbar_wait<PAIR>(bar_tempty + 8 * buf, tph ^ 1, p.status, s_abort)) return false;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      bool ok = true;
      for (int kb = 0; kb < t.nkb; ++kb) {
        if (!mbar_wait(bar_full + 8 * stage, phase, p.status, s_abort)) { ok = false; break; }
        if constexpr (C::NV)  // the converter warps have written the next f16 B tile
          if (!mbar_wait(bar_conv + 8 * ds, dphase, p.status, s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = sA0 + stage * C::A_BYTES;
        const uint32_t sB = sB0 + (C::NV ? ds : stage) * C::B_BYTES;
        int nk16 = BK / 16;  // MMA K steps of this stage
        if constexpr (C::K_GROUPED) {
          // last k-block of a problem: issue only the K steps holding rows of this problem (the
          // rows past its end within the last step arrive as zeros: the loads are bounded to it)
          const int valid = t.rows - kb * BK;
          if (valid < BK) nk16 = (valid + 15) / 16;
        }
        if (lane == 0) {
          if constexpr (C::MX) {
            // scale factors of this stage: smem atoms -> TMEM (16 columns per stage), then four
            // K = 32 block-scaled MMAs; MMA j reads byte j of each 32-bit scale word.
            const uint32_t sf = sSF0 + stage * C::SF_BYTES;
            const uint32_t sfa_t = tmem_base + C::SF_TMEM_COL + 16 * stage;
            const uint32_t sfb_t = sfa_t + 4;
            tmem_cp_32x128b_x4(sfa_t, make_sdesc_noswz(sf, 16, 128));
#pragma unroll
            for (int a = 0; a < BN / 128; ++a)
              tmem_cp_32x128b_x4(sfb_t + 4 * a, make_sdesc_noswz(sf + 512 + 512 * a, 16, 128));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = make_sdesc(sA + k * 32, 16, 1024);
              const uint64_t bd = make_sdesc(sB + k * 32, 16, 1024);
              const uint32_t idesc = C::IDESC | (static_cast<uint32_t>(k) << 29) |
                                     (static_cast<uint32_t>(k) << 4);
              umma_mxf8(d_tmem, ad, bd, idesc, sfa_t, sfb_t, (kb | k) != 0);
            }
          } else {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              if (k < nk16) {
                const uint64_t ad = C::A_MN ? make_sdesc(sA + k * 2048, 8192, 1024)
                                            : make_sdesc(sA + k * 32, 16, 1024);
                const uint64_t bd = C::B_MN ? make_sdesc(sB + k * 2048, 8192, 1024)
                                            : make_sdesc(sB + k * 32, 16, 1024);
                if constexpr (PAIR)
                  umma_bf16_pair(d_tmem, ad, bd, C::IDESC, (kb | k) != 0);
                else
                  umma_bf16(d_tmem, ad, bd, C::IDESC, (kb | k) != 0);
              }
            }
          }
          if constexpr (PAIR)
            umma_commit_pair_mc(bar_empty + 8 * stage, 3);
          else
            umma_commit(bar_empty + 8 * stage);
          if constexpr (C::NV) umma_commit(bar_dempty + 8 * ds);
        }
        __syncwarp();
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        if constexpr (C::NV)
          if (++ds == C::DEC_STAGES) { ds = 0; dphase ^= 1; }
      }
      if (!ok) return false;
      if (lane == 0) {
        if constexpr (PAIR)
          umma_commit_pair_mc(bar_tfull + 8 * buf, 3);
        else
          umma_commit(bar_tfull + 8 * buf);
      }
      __syncwarp();
      return true;
    };
    if constexpr (C::FUSED) {
      for (int it = 0;; ++it) {
        const int slot = it % kRing;
        if (!mbar_wait(bar_rfull + 8 * slot, (it / kRing) & 1, p.status, s_abort)) break;
        const int tile = s_ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_rempty + 8 * slot);
        if (tile >= ntiles) break;
        if (!mma_tile(decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank), it)) break;
      }
    } else {
      int it = 0;
      for (int tile = first; tile < ntiles && !*s_abort; tile += step, ++it)
        if (!mma_tile(decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank), it)) break;
    }
    // every MMA issued by this CTA has completed before TMEM is released
    if (lane == 0) {
      if constexpr (PAIR)
        umma_commit_pair(bar_drain);
      else
        umma_commit(bar_drain);
      volatile int no_abort = 0;
      mbar_wait(bar_drain, 0, p.status, &no_abort);
    }
    __syncwarp();
  } else if (C::NV && warp == 2 + C::EPI_WARPS + C::CONV_WARPS) {
    // raw B producer (one lane): the tiles of the MMA warp, each k-block's codes and scales by
    // bulk copies into the raw ring
    if (lane == 0) {
      int rs = 0;
      uint32_t rphase = 0;
      for (int tile = first; tile < ntiles && !*s_abort; tile += step) {
        const Tile t = decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank);
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(bar_rawempty + 8 * rs, rphase ^ 1, p.status, s_abort)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_rawfull + 8 * rs, C::SF_BYTES);
          if constexpr (C::NV) load_nv_raw<MODE, BN>(p, t, kb, sSF0 + rs * C::SF_BYTES, bar_rawfull + 8 * rs);
          if (++rs == C::RAW_STAGES) { rs = 0; rphase ^= 1; }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (C::NV && warp >= 2 + C::EPI_WARPS) {
    // converter warps: each k-block's raw B rows, once landed, decoded into the next free f16
    // tile, which is then published to the MMA (async proxy); the raw stage is released first
    const int ct = tid - 32 * (2 + C::EPI_WARPS);
    int rs = 0, ds = 0;
    uint32_t rphase = 0, dphase = 0;
    for (int tile = first; tile < ntiles && !*s_abort; tile += step) {
      const Tile t = decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank);
      bool ok = true;
      for (int kb = 0; kb < t.nkb; ++kb) {
        if (!mbar_wait(bar_rawfull + 8 * rs, rphase, p.status, s_abort) ||
            !mbar_wait(bar_dempty + 8 * ds, dphase ^ 1, p.status, s_abort)) {
          ok = false;
          break;
        }
        nv_convert_stage<BN, 32 * C::CONV_WARPS>(sSF0 + rs * C::SF_BYTES, sB0 + ds * C::B_BYTES, ct);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_rawempty + 8 * rs);
          mbar_arrive(bar_conv + 8 * ds);
        }
        if (++rs == C::RAW_STAGES) { rs = 0; rphase ^= 1; }
        if (++ds == C::DEC_STAGES) { ds = 0; dphase ^= 1; }
      }
      if (!ok) break;
    }
  } else if (warp >= 2) {
    const int q = warp & 3;  // TMEM lane quarter accessible to this warp
    const int half = (warp - 2) / 4;  // 8 epilogue warps: which column half
    const int r = q * 32 + lane;
    // the epilogue of the it-th tile of this CTA; false when a bounded wait ran out
    auto epi_tile = [&](const Tile& t, int it) -> bool {
      const int buf = it % C::NUM_ACC;
      const uint32_t tph = (it / C::NUM_ACC) & 1;
      if (!mbar_wait(bar_tfull + 8 * buf, tph, p.status, s_abort)) return false;
      tc_fence_after();
      const uint32_t tacc = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      // the staged and MXFP8 epilogues release the accumulator themselves (before their stores
      // when there is only one)
      const uint32_t stg = sSTG0 + (warp - 2) * C::STG_STRIDE;
      const uint32_t rel = PAIR ? mapa_shared(bar_tempty + 8 * buf, 0) : bar_tempty + 8 * buf;
      if constexpr (MODE == G_FWD_GUD) {
        if (t.sub == 0) {  // h (and G, U), then this warp's share of the M tile's readiness
          epilogue<G_FWD_GU, BN>(p, t, tacc, r, half);
          acc_release(rel, lane);
          const int mt0 = p.has_shared ? (p.T + BM - 1) / BM : 0;
          signal_counter(p.ready + (t.g ? mt0 + t.mt : t.mt), lane);
        } else {  // Y = router weight x (h W_down) into out3
          epilogue_rows<G_FWD_DOWN, BN>(p, p.out3, t, tacc, stg, q, half, lane, rel);
        }
      } else if constexpr (MODE == G_BWD_DW || MODE == G_BWD_DW_MX) {
        epilogue_dw<MODE, BN>(p, t, tacc, stg, q, half, lane, rel);
      } else if constexpr (C::ROW_STAGED) {
        epilogue_rows<MODE, BN>(p, p.out0, t, tacc, stg, q, half, lane, rel);
      } else if constexpr (MODE == G_FWD_GU_MX) {
        epilogue_gu_mx<BN>(p, t, tacc, r, half, rel);
      } else if constexpr (MODE == G_FWD_GU_NV) {
        epilogue_gu_nv<BN>(p, t, tacc, r);
        acc_release(rel, lane);
      } else if constexpr (MODE == G_BWD_DA_MX) {
        epilogue_da_mx<BN>(p, t, tacc, stg, q, half, lane, rel);
      } else {
        epilogue<MODE, BN>(p, t, tacc, r, half);
        acc_release(rel, lane);
      }
      return true;
    };
    if constexpr (C::FUSED) {
      for (int it = 0;; ++it) {
        const int slot = it % kRing;
        if (!mbar_wait(bar_rfull + 8 * slot, (it / kRing) & 1, p.status, s_abort)) break;
        const int tile = s_ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_rempty + 8 * slot);
        if (tile >= ntiles) break;
        if (!epi_tile(decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank), it)) break;
      }
    } else {
      int it = 0;
      for (int tile = first; tile < ntiles && !*s_abort; tile += step, ++it)
        if (!epi_tile(decode_tile<MODE, BN, PAIR>(p, s_off, s_mt, tile, rank), it)) break;
    }
  }
  __syncthreads();
  // a pair: neither CTA frees TMEM or leaves while the other may still arrive on its barriers
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// One warp per (expert, routed weight-gradient operand): the operand's map with the base moved to
// the expert's first row and the row extent cut to its rows (tensormap.replace on a shared-memory
// copy), published to emaps[e * kBoundMaps + j] for the tensor-map proxy.  Experts without rows
// are skipped (no tile loads them).
__global__ void __launch_bounds__(256) dw_bound_maps_kernel(const __grid_constant__ BoundMapParams bp) {
  __shared__ __align__(128) uint8_t smaps[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  if (i >= bp.E * kBoundMaps) return;
  const int e = i / kBoundMaps, j = i - e * kBoundMaps;
  const int r0 = bp.offsets[e], rows = bp.offsets[e + 1] - r0;
  if (rows <= 0) return;
  const uint32_t sm = smem_u32(smaps[warp]);
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(sm + 4 * lane),
               "r"(reinterpret_cast<const uint32_t*>(&bp.templ[j])[lane])
               : "memory");
  __syncwarp();
  if (lane == 0) {
    tmap_replace_address(sm, static_cast<const char*>(bp.base[j]) + (int64_t)r0 * bp.cols[j] * 2);
    tmap_replace_rows(sm, rows);
  }
  __syncwarp();
  tmap_publish(bp.emaps + i, sm);
}

cudaError_t launch_dw_bound_maps(const BoundMapParams& bp, cudaStream_t s) {
  const int n = bp.E * kBoundMaps;
  if (n == 0) return cudaSuccess;
  prof_begin("dw_bound_maps", s);
  dw_bound_maps_kernel<<<(n + 7) / 8, 256, 0, s>>>(bp);
  prof_end(s);
  return cudaGetLastError();
}

// ceil(2^32 / d): n / d == (n * m) >> 32 for every n with n * d < 2^32
static uint64_t div_magic(int64_t d) { return d > 0 ? ((uint64_t(1) << 32) + uint64_t(d) - 1) / uint64_t(d) : 0; }

// The K-grouped decode's divisors of this launch (tile counts of its tile numbering); false when
// a tile index times a divisor could reach 2^32, where the reciprocal division would not be exact.
template <int BN>
static bool set_div_magics(GemmParams& p, int64_t ntiles_single) {
  const int64_t per = 2 * (p.d / BM) * (p.F / BN) + (p.F / BM) * (p.d / BN);
  const int64_t nts = p.Fs / BN, ntf = p.F / BN, ntd = p.d / BN;
  p.router_nt = p.router_tiles > 0 ? p.router_tiles / (p.d / BM) : 1;
  p.dm_per = div_magic(per);
  p.dm_nt[0] = div_magic(nts > 0 ? nts : 1);
  p.dm_nt[1] = div_magic(ntf);
  p.dm_ntd = div_magic(ntd);
  p.dm_ntr = div_magic(p.router_nt);
  const int64_t dmax = std::max({per, nts, ntf, ntd, (int64_t)p.router_nt});
  return ntiles_single * dmax < (int64_t(1) << 32);
}

template <int MODE, int BN, bool PAIR = false>
static cudaError_t launch_one(const GemmParams& p_in, int grid, cudaStream_t s) {
  GemmParams p = p_in;
  if constexpr (Cfg<MODE, BN>::K_GROUPED) {
    const int64_t per = 2 * (p.d / BM) * (p.F / BN) + (p.F / BM) * (p.d / BN);
    const int64_t sh = p.has_shared ? 2 * (p.d / BM) * (p.Fs / BN) + (p.Fs / BM) * (p.d / BN) : 0;
    if (!set_div_magics<BN>(p, p.router_tiles + sh + (int64_t)p.E * per)) return cudaErrorInvalidValue;
  }
  constexpr int smem = smem_bytes_for<MODE, BN, PAIR>();
  static_assert(smem <= 227 * 1024, "shared memory of one CTA exceeds 227 KB");
  auto k = moe_gemm_kernel<MODE, BN, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static const char* kNames[] = {"gemm_fwd_gate_up", "gemm_fwd_down",      "gemm_bwd_da",
                                 "gemm_bwd_dx",      "gemm_bwd_dw",        "gemm_fwd_gate_up_mx",
                                 "gemm_fwd_down_mx", "gemm_bwd_da_mx",     "gemm_bwd_dx_mx",
                                 "gemm_bwd_dw_mx",   "gemm_fwd_fused",     "gemm_fwd_gate_up_nv",
                                 "gemm_fwd_down_nv"};
  if constexpr (!PAIR) {
    if (grid <= 0) return cudaSuccess;
    prof_begin(kNames[MODE], s);
    k<<<grid, Cfg<MODE, BN>::THREADS, smem, s>>>(p);
    prof_end(s);
    return cudaGetLastError();
  } else {
    // clusters of two CTAs; persistent: as many pairs as fit at once, at most one per pair tile
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(Cfg<MODE, BN>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.gridDim = dim3(2);
    // pairs resident at once: a property of this kernel on this device, queried once per device
    static int fit_of_device[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int fit = (dev >= 0 && dev < 64) ? fit_of_device[dev] : 0;
    if (fit == 0) {
      e = cudaOccupancyMaxActiveClusters(&fit, k, &cfg);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) fit_of_device[dev] = fit;
    }
    const int pairs = std::min((grid + 1) / 2, fit);
    if (pairs <= 0) return grid <= 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(2 * pairs);
    prof_begin(kNames[MODE], s);
    e = cudaLaunchKernelEx(&cfg, k, p);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
}

// Groups with at least this many M tiles (of 128 rows, or 256 in CTA pairs) run their N tiles
// fastest.  Measured on the Kimi-class forward: 10.52-10.63 -> 9.96-10.02 ms per step (the hot
// expert's and the shared expert's rows, 229 and 235 MB, no longer re-read from HBM for each of
// the 16 gate/up N tiles; the lower DRAM traffic also let the power-capped clock rise); 4 beat 8
// on the MXFP8 training step and equalled it elsewhere; 2 was slower on the DSV3 forward.
constexpr int kNFastMTiles = 4;

cudaError_t launch_gemm(int mode, int bn, const GemmParams& p_in, int grid, cudaStream_t s, bool pair) {
  GemmParams p = p_in;
  p.nfast_mt = kNFastMTiles;
  switch (mode) {
    case G_FWD_GU:
      return pair ? launch_one<G_FWD_GU, 256, true>(p, grid, s) : launch_one<G_FWD_GU, 256>(p, grid, s);
    case G_FWD_DOWN:
      if (bn != 256) return launch_one<G_FWD_DOWN, 128>(p, grid, s);
      return pair ? launch_one<G_FWD_DOWN, 256, true>(p, grid, s) : launch_one<G_FWD_DOWN, 256>(p, grid, s);
    case G_BWD_DA:
      return bn == 256 ? launch_one<G_BWD_DA, 256>(p, grid, s) : launch_one<G_BWD_DA, 128>(p, grid, s);
    case G_BWD_DX:
      return bn == 256 ? launch_one<G_BWD_DX, 256>(p, grid, s) : launch_one<G_BWD_DX, 128>(p, grid, s);
    case G_BWD_DW:
      if (bn != 256) return launch_one<G_BWD_DW, 128>(p, grid, s);
      return pair ? launch_one<G_BWD_DW, 256, true>(p, grid, s) : launch_one<G_BWD_DW, 256>(p, grid, s);
    case G_FWD_GU_MX: return launch_one<G_FWD_GU_MX, 256>(p, grid, s);
    case G_FWD_DOWN_MX: return launch_one<G_FWD_DOWN_MX, 256>(p, grid, s);
    case G_BWD_DA_MX: return launch_one<G_BWD_DA_MX, 128>(p, grid, s);  // two accumulators
    case G_BWD_DX_MX: return launch_one<G_BWD_DX_MX, 256>(p, grid, s);
    case G_BWD_DW_MX: return launch_one<G_BWD_DW_MX, 256>(p, grid, s);
    case G_FWD_GUD: return launch_one<G_FWD_GUD, 256>(p, grid, s);
    case G_FWD_GU_NV: return launch_one<G_FWD_GU_NV, 256>(p, grid, s);
    case G_FWD_DOWN_NV: return launch_one<G_FWD_DOWN_NV, 256>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mok
