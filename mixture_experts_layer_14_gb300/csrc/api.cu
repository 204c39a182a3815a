// C-ABI entry points of libmok: argument checks, workspace layout, TMA tensor maps and the
// launch sequence of each call.  Host code only; every step of the layer runs in the kernels
// of route.cu, dispatch.cu, elementwise.cu and moe_gemm.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "mok_internal.h"

namespace mok {

static thread_local int g_last_launches = 0;
static std::atomic<int> g_forward_schedule{MOK_SCHEDULE_TWO_LAUNCHES};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 (esize 2) or byte (esize 1) tensor of `rank` dims (innermost first), 128-byte swizzle,
// zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, int esize = 2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  rank, const_cast<void*>(ptr), dims,
                  strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// 2D row-major [rows, cols], box {bc, br}
static bool map2d(CUtensorMap* m, const void* p, uint64_t rows, uint64_t cols, uint32_t bc,
                  uint32_t br, int esize = 2) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t str[1] = {cols * esize};
  const uint32_t box[2] = {bc, br};
  return make_map(m, p, 2, dims, str, box, esize);
}
// 3D row-major [n, rows, cols], box {bc, br, 1}
static bool map3d(CUtensorMap* m, const void* p, uint64_t n, uint64_t rows, uint64_t cols,
                  uint32_t bc, uint32_t br, int esize = 2) {
  const uint64_t dims[3] = {cols, rows, n};
  const uint64_t str[2] = {cols * esize, rows * cols * esize};
  const uint32_t box[3] = {bc, br, 1};
  return make_map(m, p, 3, dims, str, box, esize);
}

// ------------------------------------------------------------------ checks and layouts
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_dims(const mok_dims* d) {
  if (!d) return MOK_ERR_INVALID_ARG;
  if (d->T < 0 || d->T > 0x7fffffffLL / 8) return MOK_ERR_UNSUPPORTED;
  if (d->d <= 0 || d->d % 128) return MOK_ERR_UNSUPPORTED;
  if (d->F <= 0 || d->F % 128) return MOK_ERR_UNSUPPORTED;
  if (d->n_shared != 0 && d->n_shared != 1) return MOK_ERR_UNSUPPORTED;
  if (d->n_shared == 1 && (d->F_shared <= 0 || d->F_shared % 128)) return MOK_ERR_UNSUPPORTED;
  if (d->k < 1 || d->k > kMaxK || d->E < d->k || d->E > kMaxE || d->E % 8) return MOK_ERR_UNSUPPORTED;
  if (d->dtype != MOK_BF16 && d->dtype != MOK_MXFP8 && d->dtype != MOK_NVFP4) return MOK_ERR_INVALID_ARG;
  if (d->dtype != MOK_BF16 && d->d % 256) return MOK_ERR_UNSUPPORTED;  // 256-wide down tiles
  return MOK_OK;
}

struct Layout {
  size_t off[48];
  size_t total;
};
static size_t al(size_t x) { return (x + 1023) & ~size_t(1023); }

enum FwdSlot {
  FW_STATUS, FW_HIST, FW_XS, FW_H, FW_HSH, FW_YS, FW_YSH,
  FW_SYNC,  // fused forward: work counter, then one readiness counter per M tile
  // MXFP8 only: E4M3 codes and UE8M0 scale atoms of x, x_sorted, h, h_sh
  FW_XQ, FW_XSC, FW_XQS, FW_XSCS, FW_HQ, FW_HSC, FW_HQSH, FW_HSCSH,
  FW_N
};
enum PrepSlot {  // MXFP8 prepared weights: K-major codes [n][N][K] and scale atoms
  PR_GQ, PR_GS, PR_UQ, PR_US, PR_DQ, PR_DS, PR_SGQ, PR_SGS, PR_SUQ, PR_SUS, PR_SDQ, PR_SDS, PR_N
};
enum PrepNvSlot {  // NVFP4 prepared weights: code rows, scale rows, per-matrix g, scratch, act
  PN_GQ, PN_GS, PN_UQ, PN_US, PN_DQ, PN_DS, PN_SGQ, PN_SGS, PN_SUQ, PN_SUS, PN_SDQ, PN_SDS,
  PN_G, PN_AMAX, PN_ACT, PN_N
};
enum PrepBwdSlot {  // MXFP8 backward weights: codes quantised along the backward GEMMs' K
  PB_DQ, PB_DS,    // W_down [E][F][d] along d (dY W_down^T)
  PB_GQ, PB_GS,    // W_gate [E][d][F] along F (dG W_gate^T)
  PB_UQ, PB_US,    // W_up
  PB_SDQ, PB_SDS, PB_SGQ, PB_SGS, PB_SUQ, PB_SUS,  // the shared expert's, likewise
  PB_N
};
enum BwdSlot {
  BW_STATUS, BW_DYS, BW_DG, BW_DU, BW_HW, BW_DGSH, BW_DUSH, BW_HWSH, BW_P, BW_DL,
  BW_DXS, BW_DXSH,
  BW_TMAP,  // weight-gradient GEMM: expert-bounded tensor-map copies
  // MXFP8 only.  dY codes and atoms (token order, then expert order); dG, dU codes and atoms
  // (routed, shared); the router term dl W_r^T of dX; the transposed token-axis operands of the
  // weight gradients (routed [.][128 NKB1], shared [.][128 NKB0]) with their atoms.
  BW_DYQ, BW_DYSC, BW_DYQS, BW_DYSCS,
  BW_DGQ, BW_DGSC, BW_DUQ, BW_DUSC, BW_DGQSH, BW_DGSCSH, BW_DUQSH, BW_DUSCSH,
  BW_DXR,
  BW_XT, BW_XTS, BW_DYT, BW_DYTS, BW_DGT, BW_DGTS, BW_DUT, BW_DUTS, BW_HWT, BW_HWTS,
  BW_XT0, BW_XTS0, BW_DYT0, BW_DYTS0, BW_DGT0, BW_DGTS0, BW_DUT0, BW_DUTS0, BW_HWT0, BW_HWTS0,
  BW_N
};
enum SavedSlot { SV_G, SV_U, SV_GSH, SV_USH, SV_XS, SV_N };
enum HostSlot { HS_X, HS_Y, HS_IDX, HS_W, HS_CNT, HS_OFF, HS_STOK, HS_SW, HS_INV, HS_N };

static int bn_for(int a, int b, int c) { return (a % 256 == 0 && b % 256 == 0 && c % 256 == 0) ? 256 : 128; }

static Layout layout_fwd(const mok_dims* d) {
  const int64_t T = d->T, R = T * d->k;
  const int Fs = d->n_shared ? d->F_shared : 0;
  const int64_t nblk = (T + kDispatchChunk - 1) / kDispatchChunk;
  size_t sz[FW_N] = {};
  sz[FW_STATUS] = 256;
  sz[FW_HIST] = sizeof(int32_t) * d->E * std::max<int64_t>(nblk, 1);
  sz[FW_XS] = 2ull * R * d->d;
  sz[FW_H] = 2ull * R * d->F;
  sz[FW_HSH] = 2ull * T * Fs;
  sz[FW_YS] = 2ull * R * d->d;
  sz[FW_YSH] = 2ull * T * d->d * d->n_shared;
  sz[FW_SYNC] = 256 + 4ull * ((T + BM - 1) / BM + (R + BM - 1) / BM + d->E);
  if (d->dtype == MOK_MXFP8) {
    sz[FW_XS] = 0;
    sz[FW_H] = 0;
    sz[FW_HSH] = 0;
    // scale atoms: 4 bytes per row and K block of 128, rows padded to whole M tiles; the
    // expert-ordered tensors hold at most ceil(R / 128) + E tiles
    const int64_t mt_x = (T + BM - 1) / BM, mt_r = (R + BM - 1) / BM + d->E;
    sz[FW_XQ] = 1ull * T * d->d;
    sz[FW_XSC] = 4ull * BM * mt_x * (d->d / 128);
    sz[FW_XQS] = 1ull * R * d->d;
    sz[FW_XSCS] = 4ull * BM * mt_r * (d->d / 128);
    sz[FW_HQ] = 1ull * R * d->F;
    sz[FW_HSC] = 4ull * BM * mt_r * (d->F / 128);
    sz[FW_HQSH] = 1ull * T * Fs;
    sz[FW_HSCSH] = 4ull * BM * mt_x * (Fs / 128);
  }
  if (d->dtype == MOK_NVFP4) sz[FW_XQ] = 2ull * T * d->d;  // x as f16 NVFP4 values; XS, H, HSH f16
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < FW_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

// MXFP8 weight gradients: K blocks of 128 tokens in the transposed operands (row stride / 128).
// Routed: every expert's tokens padded to whole blocks, at most ceil(R / 128) + E blocks.
static int64_t mx_nkb_routed(const mok_dims* d) { return (d->T * d->k + 127) / 128 + d->E; }
static int64_t mx_nkb_shared(const mok_dims* d) { return (d->T + 127) / 128; }

static int bwd_bn_da(const mok_dims* d) { return bn_for(d->F, d->n_shared ? d->F_shared : 256, 256); }

static Layout layout_bwd(const mok_dims* d) {
  const int64_t T = d->T, R = T * d->k;
  const int Fs = d->n_shared ? d->F_shared : 0;
  const int ldl = (d->E + 63) & ~63;
  const int ntda = d->F / bwd_bn_da(d);
  size_t sz[BW_N] = {};
  sz[BW_STATUS] = 256;
  sz[BW_DYS] = 2ull * R * d->d;
  sz[BW_DG] = sz[BW_DU] = sz[BW_HW] = 2ull * R * d->F;
  sz[BW_DGSH] = sz[BW_DUSH] = sz[BW_HWSH] = 2ull * T * Fs;
  sz[BW_P] = 4ull * R * ntda;
  sz[BW_DL] = 2ull * T * ldl;
  sz[BW_DXS] = 2ull * R * d->d;
  sz[BW_DXSH] = 2ull * T * d->d;
  sz[BW_TMAP] = sizeof(CUtensorMap) * (size_t)kBoundMaps * d->E;
  if (d->dtype == MOK_MXFP8) {
    const int64_t mt_x = (T + BM - 1) / BM, mt_r = (R + BM - 1) / BM + d->E;
    const int64_t k1 = 128 * mx_nkb_routed(d), k0 = 128 * mx_nkb_shared(d);
    sz[BW_DYS] = 0;
    sz[BW_TMAP] = 0;
    // dG, dU, w*h go straight from the dA epilogue into codes (along F and along tokens)
    sz[BW_DG] = sz[BW_DU] = sz[BW_HW] = 0;
    sz[BW_DGSH] = sz[BW_DUSH] = sz[BW_HWSH] = 0;
    sz[BW_P] = 4ull * R * (d->F / 128);
    sz[BW_DYQ] = 1ull * T * d->d;
    sz[BW_DYSC] = 4ull * BM * mt_x * (d->d / 128);
    sz[BW_DYQS] = 1ull * R * d->d;
    sz[BW_DYSCS] = 4ull * BM * mt_r * (d->d / 128);
    sz[BW_DGQ] = sz[BW_DUQ] = 1ull * R * d->F;
    sz[BW_DGSC] = sz[BW_DUSC] = 4ull * BM * mt_r * (d->F / 128);
    sz[BW_DGQSH] = sz[BW_DUQSH] = 1ull * T * Fs;
    sz[BW_DGSCSH] = sz[BW_DUSCSH] = 4ull * BM * mt_x * (Fs / 128);
    sz[BW_DXR] = 2ull * T * d->d;
    sz[BW_XT] = sz[BW_DYT] = 1ull * d->d * k1;
    sz[BW_DGT] = sz[BW_DUT] = sz[BW_HWT] = 1ull * d->F * k1;
    sz[BW_XT0] = sz[BW_DYT0] = 1ull * d->d * k0 * d->n_shared;
    sz[BW_DGT0] = sz[BW_DUT0] = sz[BW_HWT0] = 1ull * Fs * k0;
    for (int i : {BW_XT, BW_DYT, BW_DGT, BW_DUT, BW_HWT, BW_XT0, BW_DYT0, BW_DGT0, BW_DUT0, BW_HWT0})
      sz[i + 1] = sz[i] / 32;  // scale atoms: one byte per 32 codes
  }
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < BW_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

static Layout layout_prepared(const mok_dims* d) {
  const uint64_t E = d->E, dd = d->d, F = d->F, Fs = d->n_shared ? d->F_shared : 0;
  size_t sz[PR_N] = {E * F * dd, E * F * dd / 32, E * F * dd, E * F * dd / 32, E * dd * F, E * dd * F / 32,
                     Fs * dd, Fs * dd / 32, Fs * dd, Fs * dd / 32, dd * Fs, dd * Fs / 32};
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < PR_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

// NVFP4: codes 1/2 byte and scales 1/16 byte per weight element; g and amax per matrix
static Layout layout_prepared_nv(const mok_dims* d) {
  const uint64_t E = d->E, dd = d->d, F = d->F, Fs = d->n_shared ? d->F_shared : 0;
  const uint64_t nmat = 3 * E + 3;
  size_t sz[PN_N] = {E * dd * F / 2, E * dd * F / 16, E * dd * F / 2, E * dd * F / 16,
                     E * F * dd / 2, E * F * dd / 16, dd * Fs / 2, dd * Fs / 16, dd * Fs / 2,
                     dd * Fs / 16, Fs * dd / 2, Fs * dd / 16, 4 * nmat, 4 * nmat, 8};
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < PN_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

static Layout layout_prepared_bwd(const mok_dims* d) {
  const uint64_t E = d->E, dd = d->d, F = d->F, Fs = d->n_shared ? d->F_shared : 0;
  size_t sz[PB_N] = {E * F * dd, E * F * dd / 32, E * dd * F, E * dd * F / 32, E * dd * F, E * dd * F / 32,
                     Fs * dd, Fs * dd / 32, dd * Fs, dd * Fs / 32, dd * Fs, dd * Fs / 32};
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < PB_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

static Layout layout_saved(const mok_dims* d) {
  const int64_t T = d->T, R = T * d->k;
  const int Fs = d->n_shared ? d->F_shared : 0;
  // G, U, their shared-expert copies (bf16; fp32 for MXFP8, whose backward requantises the
  // values derived from them), x in expert order (bf16 weight gradients only)
  const size_t gb = d->dtype == MOK_MXFP8 ? 4 : 2;
  size_t sz[SV_N] = {gb * R * d->F, gb * R * d->F, gb * T * Fs, gb * T * Fs,
                     d->dtype == MOK_MXFP8 ? 0 : 2ull * R * d->d};
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < SV_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

static Layout layout_host(const mok_dims* d) {
  const int64_t T = d->T, R = T * d->k;
  // x: two buffers, alternating per call (see mok_layer_forward_host)
  size_t sz[HS_N] = {2 * al(2ull * T * d->d), 2ull * T * d->d, 4ull * R, 4ull * R, 4ull * d->E,
                     4ull * (d->E + 1), 4ull * R, 4ull * R, 4ull * R};
  Layout L{};
  size_t o = 0;
  for (int i = 0; i < HS_N; ++i) { L.off[i] = o; o += al(sz[i]); }
  L.total = o;
  return L;
}

template <class P>
static P at(void* base, size_t off) {
  return reinterpret_cast<P>(static_cast<char*>(base) + off);
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA; }

// MXFP8 backward (the MXFP8 reading of the layer's training step): every expert GEMM takes E4M3
// operands with UE8M0 scales along its own reduction dimension (dY and W_down along d; dG, dU,
// W_gate, W_up along F; the weight gradients' operands along each expert's tokens); the router
// terms dl W_router^T and x^T dl stay on the bf16 path.
static int backward_mxfp8(const mok_dims* dims, const mok_weights* w, const void* x, const void* dY,
                          const void* saved, const int32_t* topk_idx, const float* topk_w,
                          const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                          const int32_t* inv_pos, void* dX, void* dW_gate, void* dW_up,
                          void* dW_down, void* dWs_gate, void* dWs_up, void* dWs_down,
                          float* dlogits, void* dW_router, void* ws, cudaStream_t s,
                          int* launches) {
  if (!w->prepared_bwd || !aligned16(w->prepared_bwd)) return MOK_ERR_INVALID_ARG;
  const bool sh = dims->n_shared == 1;
  const int64_t T = dims->T, R = T * dims->k;
  const int d = dims->d, E = dims->E, F = dims->F, Fs = sh ? dims->F_shared : 0, k = dims->k;
  const Layout L = layout_bwd(dims);
  const Layout S = layout_saved(dims);
  const Layout P = layout_prepared_bwd(dims);
  auto pw = [&](int i) { return static_cast<const char*>(w->prepared_bwd) + P.off[i]; };
  auto pu8 = [&](int i) { return reinterpret_cast<const uint8_t*>(pw(i)); };
  auto W = [&](int i) { return at<void*>(ws, L.off[i]); };
  auto W8 = [&](int i) { return at<uint8_t*>(ws, L.off[i]); };
  auto SV = [&](int i) { return at<void*>(const_cast<void*>(saved), S.off[i]); };
  const int grid_cap = num_sms();
  const int64_t mt_x = (T + BM - 1) / BM, mt_rb = (R + BM - 1) / BM + E;  // M-tile bounds
  const int nkb1 = (int)mx_nkb_routed(dims), nkb0 = (int)mx_nkb_shared(dims);
  const int ldl = (E + 63) & ~63;
  float* part = at<float*>(ws, L.off[BW_P]);
  int rc;
  // 1. dY quantised along d; its codes and scale atoms pulled into expert order
  rc = cuda_status(launch_mx_quantize_rows(dY, T, d, W(BW_DYQ), W(BW_DYSC), true, s));
  if (rc == MOK_OK)
    rc = cuda_status(launch_gather_rows("gather_bytes", W(BW_DYQ), nullptr, inv_pos, T, k, d,
                                        W(BW_DYQS), nullptr, s));
  if (rc == MOK_OK)
    rc = cuda_status(launch_gather_scale_atoms(W(BW_DYSC), sorted_tok, offsets, E, T, R, d,
                                               W(BW_DYSCS), s));
  if (rc != MOK_OK) return rc;
  *launches += 3;
  // 2. a = dY W_down^T; epilogue: dG and dU quantised along F (for dX), dG, dU and w*h along
  // tokens (for the weight gradients), <a, h>
  {
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], W(BW_DYQ), T, d, 128, 128, 1);
      ok &= map3d(&p.maps[MS_B0], pw(PB_SDQ), 1, Fs, d, 128, 128, 1);
    }
    ok &= map2d(&p.maps[MS_A3], W(BW_DYQS), R, d, 128, 128, 1);
    ok &= map3d(&p.maps[MS_B3], pw(PB_DQ), E, F, d, 128, 128, 1);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = Fs / 128;  // 128-column N tiles: two accumulators, the epilogue overlaps the MMAs
    p.nt[1] = F / 128;
    p.in0[0] = SV(SV_GSH); p.in1[0] = SV(SV_USH);
    p.in0[1] = SV(SV_G); p.in1[1] = SV(SV_U);
    p.tq[0][0] = W8(BW_DGT0); p.tq[0][1] = W8(BW_DUT0); p.tq[0][2] = W8(BW_HWT0);
    p.tsc[0][0] = W8(BW_DGTS0); p.tsc[0][1] = W8(BW_DUTS0); p.tsc[0][2] = W8(BW_HWTS0);
    p.tq[1][0] = W8(BW_DGT); p.tq[1][1] = W8(BW_DUT); p.tq[1][2] = W8(BW_HWT);
    p.tsc[1][0] = W8(BW_DGTS); p.tsc[1][1] = W8(BW_DUTS); p.tsc[1][2] = W8(BW_HWTS);
    p.tnkb[0] = nkb0;
    p.tnkb[1] = nkb1;
    p.qout[0][0] = W(BW_DGQSH); p.qout[0][1] = W(BW_DUQSH);
    p.qsc[0][0] = W8(BW_DGSCSH); p.qsc[0][1] = W8(BW_DUSCSH);
    p.qout[1][0] = W(BW_DGQ); p.qout[1][1] = W(BW_DUQ);
    p.qsc[1][0] = W8(BW_DGSC); p.qsc[1][1] = W8(BW_DUSC);
    p.sfa[0][0] = W8(BW_DYSC);
    p.sfa[1][0] = W8(BW_DYSCS);
    p.sfb[0][0] = pu8(PB_SDS);
    p.sfb[1][0] = pu8(PB_DS);
    p.sf_kb[0] = p.sf_kb[1] = d / 128;
    p.row_w = sorted_w;
    p.partial = part;
    p.status = static_cast<int*>(ws);
    const int64_t bound = (sh ? mt_x * p.nt[0] : 0) + mt_rb * p.nt[1];
    rc = cuda_status(launch_gemm(G_BWD_DA_MX, 128, p, (int)std::min<int64_t>(grid_cap, bound), s));
    if (rc != MOK_OK) return rc;
    ++*launches;
  }
  // 3. router backward: dw (128-column partials of <a, h>), dlogits, bf16 dl
  rc = cuda_status(launch_router_backward(T, E, k, F / 128, topk_idx, topk_w, inv_pos, part,
                                          dlogits, W(BW_DL), s));
  if (rc != MOK_OK) return rc;
  ++*launches;
  // 4. dX_s = dG W_gate^T + dU W_up^T
  {
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], W(BW_DGQSH), T, Fs, 128, 128, 1);
      ok &= map2d(&p.maps[MS_A1], W(BW_DUQSH), T, Fs, 128, 128, 1);
      ok &= map3d(&p.maps[MS_B0], pw(PB_SGQ), 1, d, Fs, 128, 256, 1);
      ok &= map3d(&p.maps[MS_B1], pw(PB_SUQ), 1, d, Fs, 128, 256, 1);
    }
    ok &= map2d(&p.maps[MS_A3], W(BW_DGQ), R, F, 128, 128, 1);
    ok &= map2d(&p.maps[MS_A4], W(BW_DUQ), R, F, 128, 128, 1);
    ok &= map3d(&p.maps[MS_B3], pw(PB_GQ), E, d, F, 128, 256, 1);
    ok &= map3d(&p.maps[MS_B4], pw(PB_UQ), E, d, F, 128, 256, 1);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = p.nt[1] = d / 256;
    p.sfa[0][0] = W8(BW_DGSCSH); p.sfa[0][1] = W8(BW_DUSCSH);
    p.sfa[1][0] = W8(BW_DGSC); p.sfa[1][1] = W8(BW_DUSC);
    p.sfb[0][0] = pu8(PB_SGS); p.sfb[0][1] = pu8(PB_SUS);
    p.sfb[1][0] = pu8(PB_GS); p.sfb[1][1] = pu8(PB_US);
    p.sf_kb[0] = Fs / 128;
    p.sf_kb[1] = F / 128;
    p.out0[0] = W(BW_DXSH);
    p.out0[1] = W(BW_DXS);
    p.status = static_cast<int*>(ws);
    const int64_t bound = (sh ? mt_x * p.nt[0] : 0) + mt_rb * p.nt[1];
    rc = cuda_status(launch_gemm(G_BWD_DX_MX, 256, p, (int)std::min<int64_t>(grid_cap, bound), s));
    if (rc != MOK_OK) return rc;
    ++*launches;
  }
  // 5. the router term of dX, dl W_router^T (bf16 GEMM, one K segment)
  {
    GemmParams p{};
    bool ok = map2d(&p.maps[MS_A0], W(BW_DL), T, ldl, 64, 128);
    ok &= map3d(&p.maps[MS_B0], w->W_router, 1, d, E, 64, 256);
    if (!ok) return MOK_ERR_CUDA;
    p.segkb[0][0] = ldl / BK;
    p.has_shared = 1;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = d / 256;
    p.out0[0] = W(BW_DXR);
    p.status = static_cast<int*>(ws);
    rc = cuda_status(launch_gemm(G_BWD_DX, 256, p, (int)std::min<int64_t>(grid_cap, mt_x * p.nt[0]), s));
    if (rc != MOK_OK) return rc;
    ++*launches;
  }
  // 6. x and dY quantised along tokens, transposed (dG, dU and w*h came from the dA epilogue):
  // routed (rows pulled by sorted_tok), then the shared expert's (all tokens in order)
  {
    using bf = const __nv_bfloat16*;
    auto tq = [&](bf a, bf b, bf c, int slot_a, int slot_b, int slot_c, int n, int C, int64_t nsrc,
                  const int32_t* rows, const int32_t* offs, int nkb) {
      TokQuantParams tp{};
      const bf srcs[3] = {a, b, c};
      const int slots[3] = {slot_a, slot_b, slot_c};
      for (int i = 0; i < n; ++i) {
        tp.src[i] = srcs[i];
        tp.q[i] = W8(slots[i]);
        tp.sc[i] = W8(slots[i] + 1);
      }
      tp.nops = n;
      tp.C = C;
      tp.nsrc = nsrc;
      tp.rows_idx = rows;
      tp.offsets = offs;
      tp.E = E;
      tp.nkb = nkb;
      return cuda_status(launch_mx_quantize_tokens(tp, s));
    };
    const bf bx = static_cast<bf>(x), bdy = static_cast<bf>(dY);
    rc = tq(bx, bdy, nullptr, BW_XT, BW_DYT, 0, 2, d, T, sorted_tok, offsets, nkb1);
    if (rc == MOK_OK && sh) rc = tq(bx, bdy, nullptr, BW_XT0, BW_DYT0, 0, 2, d, T, nullptr, nullptr, nkb0);
    if (rc != MOK_OK) return rc;
    *launches += sh ? 2 : 1;
  }
  // 7. weight gradients: dW_gate = X^T dG, dW_up = X^T dU, dW_down = (w h)^T dY, K = tokens
  {
    GemmParams p{};
    bool ok = true;
    const uint64_t k0 = 128ull * nkb0, k1 = 128ull * nkb1;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], W(BW_XT0), d, k0, 128, 128, 1);
      ok &= map2d(&p.maps[MS_A1], W(BW_HWT0), Fs, k0, 128, 128, 1);
      ok &= map2d(&p.maps[MS_B0], W(BW_DGT0), Fs, k0, 128, 256, 1);
      ok &= map2d(&p.maps[MS_B1], W(BW_DUT0), Fs, k0, 128, 256, 1);
      ok &= map2d(&p.maps[MS_B2], W(BW_DYT0), d, k0, 128, 256, 1);
      p.sfa[0][0] = W8(BW_XTS0); p.sfa[0][1] = W8(BW_HWTS0);
      p.sfb[0][0] = W8(BW_DGTS0); p.sfb[0][1] = W8(BW_DUTS0); p.sfb[0][2] = W8(BW_DYTS0);
    }
    ok &= map2d(&p.maps[MS_A3], W(BW_XT), d, k1, 128, 128, 1);
    ok &= map2d(&p.maps[MS_A4], W(BW_HWT), F, k1, 128, 128, 1);
    ok &= map2d(&p.maps[MS_B3], W(BW_DGT), F, k1, 128, 256, 1);
    ok &= map2d(&p.maps[MS_B4], W(BW_DUT), F, k1, 128, 256, 1);
    ok &= map2d(&p.maps[MS_B5], W(BW_DYT), d, k1, 128, 256, 1);
    if (!ok) return MOK_ERR_CUDA;
    p.sfa[1][0] = W8(BW_XTS); p.sfa[1][1] = W8(BW_HWTS);
    p.sfb[1][0] = W8(BW_DGTS); p.sfb[1][1] = W8(BW_DUTS); p.sfb[1][2] = W8(BW_DYTS);
    p.sf_kb[0] = nkb0;
    p.sf_kb[1] = nkb1;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.out0[0] = dWs_gate; p.out1[0] = dWs_up; p.out2[0] = dWs_down;
    p.out0[1] = dW_gate; p.out1[1] = dW_up; p.out2[1] = dW_down;
    p.status = static_cast<int*>(ws);
    const int64_t total = (sh ? 2 * (d / BM) * (Fs / 256) + (Fs / BM) * (d / 256) : 0) +
                          (int64_t)E * (2 * (d / BM) * (F / 256) + (F / BM) * (d / 256));
    rc = cuda_status(launch_gemm(G_BWD_DW_MX, 256, p, (int)std::min<int64_t>(grid_cap, total), s));
    if (rc != MOK_OK) return rc;
    ++*launches;
  }
  // 8. the router's weight gradient x^T dl (bf16 GEMM)
  if (dW_router) {
    GemmParams p{};
    bool ok = map2d(&p.maps[MS_R_A], x, T, d, 64, 64);
    ok &= map2d(&p.maps[MS_R_B], W(BW_DL), T, ldl, 64, 64);
    if (!ok) return MOK_ERR_CUDA;
    p.router_tiles = (d / BM) * ((E + 255) / 256);
    p.E_cols = E;
    p.out_router = dW_router;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.status = static_cast<int*>(ws);
    rc = cuda_status(launch_gemm(G_BWD_DW, 256, p, std::min(grid_cap, p.router_tiles), s));
    if (rc != MOK_OK) return rc;
    ++*launches;
  }
  // 9. dX = dX_shared + dl W_router^T + routed rows in ascending expert order
  rc = cuda_status(launch_combine(T, d, k, topk_idx, inv_pos, W(BW_DXS), sh ? W(BW_DXSH) : nullptr,
                                  dX, s, W(BW_DXR)));
  if (rc != MOK_OK) return rc;
  ++*launches;
  return MOK_OK;
}

}  // namespace mok

using namespace mok;

extern "C" {

size_t mok_workspace_size(const mok_dims* dims, int pass) {
  if (check_dims(dims) != MOK_OK) return 0;
  if (pass == MOK_PASS_FORWARD) return layout_fwd(dims).total;
  if (pass == MOK_PASS_BACKWARD) return layout_bwd(dims).total;
  return 0;
}

size_t mok_saved_size(const mok_dims* dims) {
  if (check_dims(dims) != MOK_OK || dims->dtype == MOK_NVFP4) return 0;
  return layout_saved(dims).total;
}

size_t mok_prepared_size(const mok_dims* dims) {
  if (check_dims(dims) != MOK_OK) return 0;
  if (dims->dtype == MOK_NVFP4) return layout_prepared_nv(dims).total;
  return dims->dtype == MOK_MXFP8 ? layout_prepared(dims).total : 0;
}

size_t mok_layer_host_extra_size(const mok_dims* dims) {
  if (check_dims(dims) != MOK_OK) return 0;
  return layout_host(dims).total;
}

// NVFP4 weights: per-matrix amax, then code and scale rows (nv.cu); the calibrated activation
// amaxes start at 0 (tensor scale 1)
static int prepare_weights_nv(const mok_dims* dims, const mok_weights* w, void* prepared,
                              cudaStream_t s) {
  const Layout P = layout_prepared_nv(dims);
  const int d = dims->d, F = dims->F, Fs = dims->F_shared, E = dims->E;
  auto q = [&](int i) { return static_cast<char*>(prepared) + P.off[i]; };
  uint32_t* amax = reinterpret_cast<uint32_t*>(q(PN_AMAX));
  float* g = reinterpret_cast<float*>(q(PN_G));
  cudaError_t e = cudaMemsetAsync(amax, 0, 4ull * (3 * E + 3), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(q(PN_ACT), 0, 8, s);
  // gate/up [E][d][F] (K = d); down [E][F][d] (K = F)
  if (e == cudaSuccess) e = launch_nv_prepare(w->W_gate, E, d, F, amax, q(PN_GQ), q(PN_GS), g, s);
  if (e == cudaSuccess) e = launch_nv_prepare(w->W_up, E, d, F, amax + E, q(PN_UQ), q(PN_US), g + E, s);
  if (e == cudaSuccess)
    e = launch_nv_prepare(w->W_down, E, F, d, amax + 2 * E, q(PN_DQ), q(PN_DS), g + 2 * E, s);
  if (dims->n_shared) {
    if (e == cudaSuccess)
      e = launch_nv_prepare(w->Ws_gate, 1, d, Fs, amax + 3 * E, q(PN_SGQ), q(PN_SGS), g + 3 * E, s);
    if (e == cudaSuccess)
      e = launch_nv_prepare(w->Ws_up, 1, d, Fs, amax + 3 * E + 1, q(PN_SUQ), q(PN_SUS), g + 3 * E + 1, s);
    if (e == cudaSuccess)
      e = launch_nv_prepare(w->Ws_down, 1, Fs, d, amax + 3 * E + 2, q(PN_SDQ), q(PN_SDS), g + 3 * E + 2, s);
  }
  if (e != cudaSuccess) return MOK_ERR_CUDA;
  g_last_launches = 2 * (dims->n_shared ? 6 : 3);
  return MOK_OK;
}

int mok_nvfp4_set_activation_amax(const mok_dims* dims, void* prepared, float amax_x, float amax_h,
                                  mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  g_last_launches = 0;
  if (dims->dtype != MOK_NVFP4 || !prepared || !aligned16(prepared)) return MOK_ERR_INVALID_ARG;
  if (!(amax_x >= 0.0f && amax_x <= 3.0e38f) || !(amax_h >= 0.0f && amax_h <= 3.0e38f))
    return MOK_ERR_INVALID_ARG;  // also rejects NaN
  const Layout P = layout_prepared_nv(dims);
  float* act = reinterpret_cast<float*>(static_cast<char*>(prepared) + P.off[PN_ACT]);
  if (launch_nv_set_act(act, amax_x, amax_h, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOK_ERR_CUDA;
  g_last_launches = 1;
  return MOK_OK;
}

int mok_prepare_weights(const mok_dims* dims, const mok_weights* w, void* prepared,
                        mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!w) return MOK_ERR_INVALID_ARG;
  g_last_launches = 0;
  if (dims->dtype == MOK_BF16) return MOK_OK;
  if (!prepared || !w->W_gate || !w->W_up || !w->W_down) return MOK_ERR_INVALID_ARG;
  if (dims->n_shared && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)) return MOK_ERR_INVALID_ARG;
  if (!aligned16(prepared)) return MOK_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dims->dtype == MOK_NVFP4) return prepare_weights_nv(dims, w, prepared, s);
  const Layout P = layout_prepared(dims);
  const int d = dims->d, F = dims->F, Fs = dims->F_shared, E = dims->E;
  auto q = [&](int i) { return static_cast<char*>(prepared) + P.off[i]; };
  // gate/up [E][d][F] -> [E][F][d] (K = d); down [E][F][d] -> [E][d][F] (K = F)
  cudaError_t e = launch_mx_quantize_transpose(w->W_gate, E, d, F, q(PR_GQ), q(PR_GS), s);
  if (e == cudaSuccess) e = launch_mx_quantize_transpose(w->W_up, E, d, F, q(PR_UQ), q(PR_US), s);
  if (e == cudaSuccess) e = launch_mx_quantize_transpose(w->W_down, E, F, d, q(PR_DQ), q(PR_DS), s);
  if (dims->n_shared) {
    if (e == cudaSuccess) e = launch_mx_quantize_transpose(w->Ws_gate, 1, d, Fs, q(PR_SGQ), q(PR_SGS), s);
    if (e == cudaSuccess) e = launch_mx_quantize_transpose(w->Ws_up, 1, d, Fs, q(PR_SUQ), q(PR_SUS), s);
    if (e == cudaSuccess) e = launch_mx_quantize_transpose(w->Ws_down, 1, Fs, d, q(PR_SDQ), q(PR_SDS), s);
  }
  if (e != cudaSuccess) return MOK_ERR_CUDA;
  g_last_launches = dims->n_shared ? 6 : 3;
  return MOK_OK;
}

size_t mok_prepared_bwd_size(const mok_dims* dims) {
  if (check_dims(dims) != MOK_OK) return 0;
  return dims->dtype == MOK_MXFP8 ? layout_prepared_bwd(dims).total : 0;
}

int mok_prepare_weights_bwd(const mok_dims* dims, const mok_weights* w, void* prepared_bwd,
                            mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!w) return MOK_ERR_INVALID_ARG;
  g_last_launches = 0;
  if (dims->dtype != MOK_MXFP8) return MOK_OK;
  if (!prepared_bwd || !w->W_gate || !w->W_up || !w->W_down) return MOK_ERR_INVALID_ARG;
  if (dims->n_shared && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)) return MOK_ERR_INVALID_ARG;
  if (!aligned16(prepared_bwd)) return MOK_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Layout P = layout_prepared_bwd(dims);
  const int64_t d = dims->d, F = dims->F, Fs = dims->F_shared, E = dims->E;
  auto q = [&](int i) { return static_cast<char*>(prepared_bwd) + P.off[i]; };
  // each weight's rows are already K-major for the backward GEMM that reads it:
  // W_down [E][F][d] rows along d; W_gate, W_up [E][d][F] rows along F
  cudaError_t e = launch_mx_quantize_rows(w->W_down, E * F, (int)d, q(PB_DQ), q(PB_DS), true, s);
  if (e == cudaSuccess) e = launch_mx_quantize_rows(w->W_gate, E * d, (int)F, q(PB_GQ), q(PB_GS), true, s);
  if (e == cudaSuccess) e = launch_mx_quantize_rows(w->W_up, E * d, (int)F, q(PB_UQ), q(PB_US), true, s);
  if (dims->n_shared) {
    if (e == cudaSuccess) e = launch_mx_quantize_rows(w->Ws_down, Fs, (int)d, q(PB_SDQ), q(PB_SDS), true, s);
    if (e == cudaSuccess) e = launch_mx_quantize_rows(w->Ws_gate, d, (int)Fs, q(PB_SGQ), q(PB_SGS), true, s);
    if (e == cudaSuccess) e = launch_mx_quantize_rows(w->Ws_up, d, (int)Fs, q(PB_SUQ), q(PB_SUS), true, s);
  }
  if (e != cudaSuccess) return MOK_ERR_CUDA;
  g_last_launches = dims->n_shared ? 6 : 3;
  return MOK_OK;
}

int mok_mx_quantize_rows(int64_t rows, int K, const void* src, void* q, void* scales,
                         mok_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 128) return MOK_ERR_UNSUPPORTED;
  if (rows > 0 && (!src || !q || !scales)) return MOK_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(q) || !aligned16(scales)) return MOK_ERR_UNSUPPORTED;
  g_last_launches = rows > 0 ? 1 : 0;
  return cuda_status(
      launch_mx_quantize_rows(src, rows, K, q, scales, false, reinterpret_cast<cudaStream_t>(stream)));
}

const char* mok_status_string(int s) {
  switch (s) {
    case MOK_OK: return "MOK_OK";
    case MOK_ERR_INVALID_ARG: return "MOK_ERR_INVALID_ARG: null pointer, negative size or bad enum";
    case MOK_ERR_UNSUPPORTED: return "MOK_ERR_UNSUPPORTED: shape or alignment outside the preconditions";
    case MOK_ERR_WORKSPACE: return "MOK_ERR_WORKSPACE: workspace too small";
    case MOK_ERR_CUDA: return "MOK_ERR_CUDA: a CUDA call failed";
    case MOK_ERR_TIMEOUT: return "MOK_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case MOK_ERR_DEVICE_CHECK: return "MOK_ERR_DEVICE_CHECK: an index failed a device-side range check";
    default: return "unknown mok status";
  }
}

int mok_read_device_status(const void* ws, int* status_out, mok_stream_t stream) {
  if (!ws || !status_out) return MOK_ERR_INVALID_ARG;
  int v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOK_ERR_CUDA;
  *status_out = v;
  return MOK_OK;
}

int mok_clear_device_status(void* ws, mok_stream_t stream) {
  if (!ws) return MOK_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)));
}

int mok_last_launch_count(void) { return g_last_launches; }

int mok_set_forward_schedule(int schedule, int* previous) {
  if (schedule != MOK_SCHEDULE_TWO_LAUNCHES && schedule != MOK_SCHEDULE_FUSED) return MOK_ERR_INVALID_ARG;
  const int old = g_forward_schedule.exchange(schedule);
  if (previous) *previous = old;
  return MOK_OK;
}

int mok_route(const mok_dims* dims, const void* x, const void* W_router, const float* bias,
              int32_t* topk_idx, float* topk_w, float* logits, void* ws, size_t ws_bytes,
              mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!ws || (dims->T > 0 && (!x || !W_router || !topk_idx || !topk_w))) return MOK_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_router) || !aligned16(ws)) return MOK_ERR_UNSUPPORTED;
  if (ws_bytes < layout_fwd(dims).total) return MOK_ERR_WORKSPACE;
  g_last_launches = 0;
  if (dims->T == 0) return MOK_OK;
  RouteParams p{};
  if (!map2d(&p.map_x, x, dims->T, dims->d, 64, 128)) return MOK_ERR_CUDA;
  if (!map2d(&p.map_w, W_router, dims->d, dims->E, 64, 64)) return MOK_ERR_CUDA;
  p.bias = bias;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.logits = logits;
  p.T = (int)dims->T;
  p.d = dims->d;
  p.E = dims->E;
  p.k = dims->k;
  p.status = static_cast<int*>(ws);
  p.splits = route_splits(dims->T, dims->d);
  rc = cuda_status(launch_route(p, reinterpret_cast<cudaStream_t>(stream)));
  if (rc == MOK_OK) g_last_launches = 1;
  return rc;
}

int mok_dispatch_index(const mok_dims* dims, const int32_t* topk_idx, const float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* sorted_tok, float* sorted_w,
                       int32_t* inv_pos, void* ws, size_t ws_bytes, mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!ws || !counts || !offsets || (dims->T > 0 && (!topk_idx || !topk_w || !sorted_tok || !sorted_w || !inv_pos)))
    return MOK_ERR_INVALID_ARG;
  if (ws_bytes < layout_fwd(dims).total) return MOK_ERR_WORKSPACE;
  g_last_launches = 0;
  const Layout L = layout_fwd(dims);
  int n = 0;
  rc = cuda_status(launch_dispatch(dims->T, dims->E, dims->k, topk_idx, topk_w, counts, offsets,
                                   sorted_tok, sorted_w, inv_pos, at<int32_t*>(ws, L.off[FW_HIST]),
                                   static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream), &n));
  if (rc == MOK_OK) g_last_launches = n;
  return rc;
}

int mok_moe_forward(const mok_dims* dims, const mok_weights* w, const void* x,
                    const int32_t* topk_idx, const int32_t* offsets, const int32_t* sorted_tok,
                    const float* sorted_w, const int32_t* inv_pos, void* y, void* saved, void* ws,
                    size_t ws_bytes, mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!w || !ws) return MOK_ERR_INVALID_ARG;
  if (dims->T == 0) {
    g_last_launches = 0;
    return ws_bytes < layout_fwd(dims).total ? MOK_ERR_WORKSPACE : MOK_OK;
  }
  if (!y || !x || !topk_idx || !offsets || !sorted_tok || !sorted_w || !inv_pos)
    return MOK_ERR_INVALID_ARG;
  if (!w->W_gate || !w->W_up || !w->W_down) return MOK_ERR_INVALID_ARG;
  if (dims->n_shared && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)) return MOK_ERR_INVALID_ARG;
  const void* ptrs[] = {x, y, saved, ws, w->W_gate, w->W_up, w->W_down, w->Ws_gate, w->Ws_up, w->Ws_down};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MOK_ERR_UNSUPPORTED;
  const Layout L = layout_fwd(dims);
  if (ws_bytes < L.total) return MOK_ERR_WORKSPACE;
  g_last_launches = 0;
  if (dims->T == 0) return MOK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t T = dims->T, R = T * dims->k;
  const int d = dims->d, E = dims->E, F = dims->F, Fs = dims->n_shared ? dims->F_shared : 0;
  const bool sh = dims->n_shared == 1;
  void* xs = at<void*>(ws, L.off[FW_XS]);
  void* h = at<void*>(ws, L.off[FW_H]);
  void* hsh = at<void*>(ws, L.off[FW_HSH]);
  void* Ys = at<void*>(ws, L.off[FW_YS]);
  void* Ysh = at<void*>(ws, L.off[FW_YSH]);
  const Layout S = layout_saved(dims);
  int launches = 0;
  const int grid_cap0 = num_sms();

  if (dims->dtype == MOK_NVFP4) {
    // NVFP4 path: x quantised once with its calibrated amax (f16 NVFP4 values), pulled into
    // expert order, the gate/up GEMM decoding the NVFP4 weights in shared memory and quantising h
    // in its epilogue, the down GEMM likewise with the router weight, and the same combine.
    if (saved) return MOK_ERR_UNSUPPORTED;
    if (!w->prepared || !aligned16(w->prepared)) return MOK_ERR_INVALID_ARG;
    const Layout P = layout_prepared_nv(dims);
    auto pw = [&](int i) { return reinterpret_cast<const uint8_t*>(w->prepared) + P.off[i]; };
    const float* g = reinterpret_cast<const float*>(pw(PN_G));
    const float* act = reinterpret_cast<const float*>(pw(PN_ACT));
    void* xq = at<void*>(ws, L.off[FW_XQ]);
    rc = cuda_status(launch_nv_quantize_act(x, T, d, act, xq, s));
    if (rc == MOK_OK)
      rc = cuda_status(launch_gather_rows("gather", xq, nullptr, inv_pos, T, dims->k, 2 * d, xs, nullptr, s));
    if (rc != MOK_OK) return rc;
    launches += 2;
    auto common = [&](GemmParams& p) {
      p.offsets = offsets;
      p.E = E;
      p.has_shared = sh;
      p.T = (int)T;
      p.d = d;
      p.F = F;
      p.Fs = Fs;
      p.nv_act = act;
      p.status = static_cast<int*>(ws);
    };
    {
      GemmParams p{};
      bool ok = true;
      if (sh) ok &= map2d(&p.maps[MS_A0], xq, T, d, 64, 128) && map2d(&p.maps[MS_A1], xq, T, d, 64, kNvSmallRows);
      ok &= map2d(&p.maps[MS_A3], xs, R, d, 64, 128) && map2d(&p.maps[MS_A4], xs, R, d, 64, kNvSmallRows);
      if (!ok) return MOK_ERR_CUDA;
      common(p);
      p.nt[0] = Fs / 128;
      p.nt[1] = F / 128;
      p.out0[0] = hsh;
      p.out0[1] = h;
      p.nvq[0][0] = pw(PN_SGQ);
      p.nvq[0][1] = pw(PN_SUQ);
      p.nvs[0][0] = pw(PN_SGS);
      p.nvs[0][1] = pw(PN_SUS);
      p.nvg[0][0] = g + 3 * E;
      p.nvg[0][1] = g + 3 * E + 1;
      p.nvq[1][0] = pw(PN_GQ);
      p.nvq[1][1] = pw(PN_UQ);
      p.nvs[1][0] = pw(PN_GS);
      p.nvs[1][1] = pw(PN_US);
      p.nvg[1][0] = g;
      p.nvg[1][1] = g + E;
      const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
      rc = cuda_status(launch_gemm(G_FWD_GU_NV, 256, p, (int)std::min<int64_t>(grid_cap0, bound), s));
      if (rc != MOK_OK) return rc;
      ++launches;
    }
    {
      GemmParams p{};
      bool ok = true;
      if (sh) ok &= map2d(&p.maps[MS_A0], hsh, T, Fs, 64, 128) && map2d(&p.maps[MS_A1], hsh, T, Fs, 64, kNvSmallRows);
      ok &= map2d(&p.maps[MS_A3], h, R, F, 64, 128) && map2d(&p.maps[MS_A4], h, R, F, 64, kNvSmallRows);
      if (!ok) return MOK_ERR_CUDA;
      common(p);
      p.nt[0] = d / 256;
      p.nt[1] = d / 256;
      p.out0[0] = Ysh;
      p.out0[1] = Ys;
      p.row_w = sorted_w;
      p.nvq[0][0] = pw(PN_SDQ);
      p.nvs[0][0] = pw(PN_SDS);
      p.nvg[0][0] = g + 3 * E + 2;
      p.nvq[1][0] = pw(PN_DQ);
      p.nvs[1][0] = pw(PN_DS);
      p.nvg[1][0] = g + 2 * E;
      const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
      rc = cuda_status(launch_gemm(G_FWD_DOWN_NV, 256, p, (int)std::min<int64_t>(grid_cap0, bound), s));
      if (rc != MOK_OK) return rc;
      ++launches;
    }
    rc = cuda_status(launch_combine(T, d, dims->k, topk_idx, inv_pos, Ys, sh ? Ysh : nullptr, y, s));
    if (rc != MOK_OK) return rc;
    g_last_launches = launches + 1;
    return MOK_OK;
  }

  if (dims->dtype == MOK_MXFP8) {
    // MXFP8 path: x quantised once (E4M3 + UE8M0 per 32 along d), its codes and scale rows
    // pulled into expert order, block-scaled gate/up GEMM whose epilogue quantises h along F,
    // block-scaled down GEMM with the router weight, and the same bf16 combine.
    if (!w->prepared || !aligned16(w->prepared)) return MOK_ERR_INVALID_ARG;
    const Layout P = layout_prepared(dims);
    auto pw = [&](int i) { return static_cast<const char*>(w->prepared) + P.off[i]; };
    void* xq = at<void*>(ws, L.off[FW_XQ]);
    uint8_t* xsc = at<uint8_t*>(ws, L.off[FW_XSC]);
    void* xqs = at<void*>(ws, L.off[FW_XQS]);
    uint8_t* xscs = at<uint8_t*>(ws, L.off[FW_XSCS]);
    void* hq = at<void*>(ws, L.off[FW_HQ]);
    uint8_t* hsc = at<uint8_t*>(ws, L.off[FW_HSC]);
    void* hqsh = at<void*>(ws, L.off[FW_HQSH]);
    uint8_t* hscsh = at<uint8_t*>(ws, L.off[FW_HSCSH]);
    rc = cuda_status(launch_mx_quantize_rows(x, T, d, xq, xsc, true, s));
    if (rc == MOK_OK)
      rc = cuda_status(launch_gather_rows("gather_bytes", xq, nullptr, inv_pos, T, dims->k, d, xqs,
                                          nullptr, s));
    if (rc == MOK_OK)
      rc = cuda_status(launch_gather_scale_atoms(xsc, sorted_tok, offsets, E, T, R, d, xscs, s));
    if (rc != MOK_OK) return rc;
    launches += 3;
    {
      GemmParams p{};
      bool ok = true;
      if (sh) {
        ok &= map2d(&p.maps[MS_A0], xq, T, d, 128, 128, 1);
        ok &= map3d(&p.maps[MS_B0], pw(PR_SGQ), 1, Fs, d, 128, 128, 1);
        ok &= map3d(&p.maps[MS_B1], pw(PR_SUQ), 1, Fs, d, 128, 128, 1);
      }
      ok &= map2d(&p.maps[MS_A3], xqs, R, d, 128, 128, 1);
      ok &= map3d(&p.maps[MS_B3], pw(PR_GQ), E, F, d, 128, 128, 1);
      ok &= map3d(&p.maps[MS_B4], pw(PR_UQ), E, F, d, 128, 128, 1);
      if (!ok) return MOK_ERR_CUDA;
      p.offsets = offsets;
      p.E = E;
      p.has_shared = sh;
      p.T = (int)T;
      p.d = d;
      p.F = F;
      p.Fs = Fs;
      p.nt[0] = Fs / 128;
      p.nt[1] = F / 128;
      p.out0[0] = hqsh;
      p.out1[0] = hscsh;
      p.out0[1] = hq;
      p.out1[1] = hsc;
      if (saved) {  // training: G and U in fp32 for the backward
        p.out2[0] = at<void*>(saved, S.off[SV_GSH]);
        p.out3[0] = at<void*>(saved, S.off[SV_USH]);
        p.out2[1] = at<void*>(saved, S.off[SV_G]);
        p.out3[1] = at<void*>(saved, S.off[SV_U]);
      }
      p.sfa[0][0] = xsc;
      p.sfa[1][0] = xscs;
      p.sfb[0][0] = reinterpret_cast<const uint8_t*>(pw(PR_SGS));
      p.sfb[0][1] = reinterpret_cast<const uint8_t*>(pw(PR_SUS));
      p.sfb[1][0] = reinterpret_cast<const uint8_t*>(pw(PR_GS));
      p.sfb[1][1] = reinterpret_cast<const uint8_t*>(pw(PR_US));
      p.sf_kb[0] = p.sf_kb[1] = d / 128;
      p.status = static_cast<int*>(ws);
      const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
      rc = cuda_status(launch_gemm(G_FWD_GU_MX, 256, p, (int)std::min<int64_t>(grid_cap0, bound), s));
      if (rc != MOK_OK) return rc;
      ++launches;
    }
    {
      GemmParams p{};
      bool ok = true;
      if (sh) {
        ok &= map2d(&p.maps[MS_A0], hqsh, T, Fs, 128, 128, 1);
        ok &= map3d(&p.maps[MS_B0], pw(PR_SDQ), 1, d, Fs, 128, 256, 1);
      }
      ok &= map2d(&p.maps[MS_A3], hq, R, F, 128, 128, 1);
      ok &= map3d(&p.maps[MS_B3], pw(PR_DQ), E, d, F, 128, 256, 1);
      if (!ok) return MOK_ERR_CUDA;
      p.offsets = offsets;
      p.E = E;
      p.has_shared = sh;
      p.T = (int)T;
      p.d = d;
      p.F = F;
      p.Fs = Fs;
      p.nt[0] = d / 256;
      p.nt[1] = d / 256;
      p.out0[0] = Ysh;
      p.out0[1] = Ys;
      p.row_w = sorted_w;
      p.sfa[0][0] = hscsh;
      p.sfa[1][0] = hsc;
      p.sfb[0][0] = reinterpret_cast<const uint8_t*>(pw(PR_SDS));
      p.sfb[1][0] = reinterpret_cast<const uint8_t*>(pw(PR_DS));
      p.sf_kb[0] = Fs / 128;
      p.sf_kb[1] = F / 128;
      p.status = static_cast<int*>(ws);
      const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
      rc = cuda_status(launch_gemm(G_FWD_DOWN_MX, 256, p, (int)std::min<int64_t>(grid_cap0, bound), s));
      if (rc != MOK_OK) return rc;
      ++launches;
    }
    rc = cuda_status(launch_combine(T, d, dims->k, topk_idx, inv_pos, Ys, sh ? Ysh : nullptr, y, s));
    if (rc != MOK_OK) return rc;
    g_last_launches = launches + 1;
    return MOK_OK;
  }

  // 1. pull-gather of every expert's token rows (into `saved` when the backward will need them)
  if (saved) xs = at<void*>(saved, S.off[SV_XS]);
  rc = cuda_status(launch_gather_rows("gather", x, nullptr, inv_pos, T, dims->k, 2 * d, xs, nullptr, s));
  if (rc != MOK_OK) return rc;
  ++launches;

  const int grid_cap = num_sms();
  // CTA pairs (256-row tiles, each SM staging half the weight columns) pay only when the experts
  // hold enough rows to fill them: measured faster at about 340 routed rows per expert, slower
  // (gate/up) at 256, where ragged experts leave many pair tiles half empty
  const bool pair = R >= 320 * (int64_t)E;
  if (!pair && d % 256 == 0 && g_forward_schedule.load() == MOK_SCHEDULE_FUSED) {
    // 2+3. gate/up and down in one persistent launch (work counter, per-M-tile readiness)
    int* sync = at<int*>(ws, L.off[FW_SYNC]);
    rc = cuda_status(cudaMemsetAsync(sync, 0, 256 + 4ull * ((T + BM - 1) / BM + (R + BM - 1) / BM + E), s));
    if (rc != MOK_OK) return rc;
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], x, T, d, 64, 128);
      ok &= map3d(&p.maps[MS_B0], w->Ws_gate, 1, d, Fs, 64, 64);
      ok &= map3d(&p.maps[MS_B1], w->Ws_up, 1, d, Fs, 64, 64);
      ok &= map2d(&p.maps[MS_A1], hsh, T, Fs, 64, 128);
      ok &= map3d(&p.maps[MS_B2], w->Ws_down, 1, Fs, d, 64, 64);
    }
    ok &= map2d(&p.maps[MS_A3], xs, R, d, 64, 128);
    ok &= map3d(&p.maps[MS_B3], w->W_gate, E, d, F, 64, 64);
    ok &= map3d(&p.maps[MS_B4], w->W_up, E, d, F, 64, 64);
    ok &= map2d(&p.maps[MS_A4], h, R, F, 64, 128);
    ok &= map3d(&p.maps[MS_B5], w->W_down, E, F, d, 64, 64);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = Fs / 128;
    p.nt[1] = F / 128;
    p.ntb[0] = p.ntb[1] = d / 256;
    p.out0[0] = hsh;
    p.out0[1] = h;
    if (saved) {
      p.out1[0] = at<void*>(saved, S.off[SV_GSH]);
      p.out2[0] = at<void*>(saved, S.off[SV_USH]);
      p.out1[1] = at<void*>(saved, S.off[SV_G]);
      p.out2[1] = at<void*>(saved, S.off[SV_U]);
    }
    p.out3[0] = Ysh;
    p.out3[1] = Ys;
    p.row_w = sorted_w;
    p.work = sync;
    p.ready = sync + 64;
    p.status = static_cast<int*>(ws);
    const int64_t mtb = (sh ? (T + BM - 1) / BM : 0) + (R + BM - 1) / BM + E;
    const int grid = (int)std::min<int64_t>(grid_cap, mtb * (F / 128 + d / 256));
    rc = cuda_status(launch_gemm(G_FWD_GUD, 256, p, grid, s));
    if (rc != MOK_OK) return rc;
    ++launches;
    rc = cuda_status(launch_combine(T, d, dims->k, topk_idx, inv_pos, Ys, sh ? Ysh : nullptr, y, s));
    if (rc != MOK_OK) return rc;
    g_last_launches = launches + 1;
    return MOK_OK;
  }
  // 2. gate/up GEMM with SiLU(gate)*up fused in the epilogue
  {
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], x, T, d, 64, 128);
      ok &= map3d(&p.maps[MS_B0], w->Ws_gate, 1, d, Fs, 64, 64);
      ok &= map3d(&p.maps[MS_B1], w->Ws_up, 1, d, Fs, 64, 64);
    }
    ok &= map2d(&p.maps[MS_A3], xs, R, d, 64, 128);
    ok &= map3d(&p.maps[MS_B3], w->W_gate, E, d, F, 64, 64);
    ok &= map3d(&p.maps[MS_B4], w->W_up, E, d, F, 64, 64);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = Fs / 128;
    p.nt[1] = F / 128;
    p.out0[0] = hsh;
    p.out0[1] = h;
    if (saved) {
      p.out1[0] = at<void*>(saved, S.off[SV_GSH]);
      p.out2[0] = at<void*>(saved, S.off[SV_USH]);
      p.out1[1] = at<void*>(saved, S.off[SV_G]);
      p.out2[1] = at<void*>(saved, S.off[SV_U]);
    }
    p.status = static_cast<int*>(ws);
    const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
    const int grid = (int)std::min<int64_t>(grid_cap, bound);
    rc = cuda_status(launch_gemm(G_FWD_GU, 256, p, grid, s, pair));
    if (rc != MOK_OK) return rc;
    ++launches;
  }
  // 3. down GEMM with the router weight fused in the epilogue
  {
    const int bn = bn_for(d, 256, 256);
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], hsh, T, Fs, 64, 128);
      ok &= map3d(&p.maps[MS_B0], w->Ws_down, 1, Fs, d, 64, 64);
    }
    ok &= map2d(&p.maps[MS_A3], h, R, F, 64, 128);
    ok &= map3d(&p.maps[MS_B3], w->W_down, E, F, d, 64, 64);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = d / bn;
    p.nt[1] = d / bn;
    p.out0[0] = Ysh;
    p.out0[1] = Ys;
    p.row_w = sorted_w;
    p.status = static_cast<int*>(ws);
    const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
    const int grid = (int)std::min<int64_t>(grid_cap, bound);
    rc = cuda_status(launch_gemm(G_FWD_DOWN, bn, p, grid, s, pair));
    if (rc != MOK_OK) return rc;
    ++launches;
  }
  // 4. fixed-order combine
  rc = cuda_status(launch_combine(T, d, dims->k, topk_idx, inv_pos, Ys, sh ? Ysh : nullptr, y, s));
  if (rc != MOK_OK) return rc;
  ++launches;
  g_last_launches = launches;
  return MOK_OK;
}

int mok_moe_backward(const mok_dims* dims, const mok_weights* w, const void* x, const void* dY,
                     const void* saved, const int32_t* topk_idx, const float* topk_w,
                     const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                     const int32_t* inv_pos, void* dX, void* dW_gate, void* dW_up, void* dW_down,
                     void* dWs_gate, void* dWs_up, void* dWs_down, float* dlogits,
                     void* dW_router, void* ws, size_t ws_bytes, mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (dims->dtype == MOK_NVFP4) return MOK_ERR_UNSUPPORTED;  // the NVFP4 variant is forward only
  if (!w || !ws || !dW_gate || !dW_up || !dW_down) return MOK_ERR_INVALID_ARG;
  if (dims->T > 0 && (!x || !dY || !saved || !topk_idx || !topk_w || !offsets || !sorted_tok ||
                      !sorted_w || !inv_pos || !dX || !dlogits))
    return MOK_ERR_INVALID_ARG;
  if (!w->W_router || !w->W_gate || !w->W_up || !w->W_down) return MOK_ERR_INVALID_ARG;
  const bool sh = dims->n_shared == 1;
  if (sh && (!w->Ws_gate || !w->Ws_up || !w->Ws_down || !dWs_gate || !dWs_up || !dWs_down))
    return MOK_ERR_INVALID_ARG;
  const void* ptrs[] = {x, dY, saved, ws, dX, dW_gate, dW_up, dW_down, dWs_gate, dWs_up, dWs_down,
                        dW_router, w->W_router, w->W_gate, w->W_up, w->W_down, w->Ws_gate, w->Ws_up,
                        w->Ws_down};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MOK_ERR_UNSUPPORTED;
  const Layout L = layout_bwd(dims);
  if (ws_bytes < L.total) return MOK_ERR_WORKSPACE;
  g_last_launches = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t T = dims->T, R = T * dims->k;
  const int d = dims->d, E = dims->E, F = dims->F, Fs = sh ? dims->F_shared : 0;
  int launches = 0;
  if (T == 0) {
    // no tokens: every weight gradient is zero
    rc = cuda_status(cudaMemsetAsync(dW_gate, 0, 2ull * E * d * F, s));
    if (rc == MOK_OK) rc = cuda_status(cudaMemsetAsync(dW_up, 0, 2ull * E * d * F, s));
    if (rc == MOK_OK) rc = cuda_status(cudaMemsetAsync(dW_down, 0, 2ull * E * d * F, s));
    if (rc == MOK_OK && sh) rc = cuda_status(cudaMemsetAsync(dWs_gate, 0, 2ull * d * Fs, s));
    if (rc == MOK_OK && sh) rc = cuda_status(cudaMemsetAsync(dWs_up, 0, 2ull * d * Fs, s));
    if (rc == MOK_OK && sh) rc = cuda_status(cudaMemsetAsync(dWs_down, 0, 2ull * d * Fs, s));
    if (rc == MOK_OK && dW_router) rc = cuda_status(cudaMemsetAsync(dW_router, 0, 2ull * d * E, s));
    return rc;
  }
  if (dims->dtype == MOK_MXFP8) {
    if (F % 256 || (sh && Fs % 256)) return MOK_ERR_UNSUPPORTED;  // 256-column tiles along F
    // the token-axis quantiser numbers its 128 x 64 tiles (x and dY) in an int
    if (2 * mx_nkb_routed(dims) * (d / 64) > 0x7fffffffLL) return MOK_ERR_UNSUPPORTED;
    rc = backward_mxfp8(dims, w, x, dY, saved, topk_idx, topk_w, offsets, sorted_tok, sorted_w,
                        inv_pos, dX, dW_gate, dW_up, dW_down, dWs_gate, dWs_up, dWs_down, dlogits,
                        dW_router, ws, s, &launches);
    if (rc == MOK_OK) g_last_launches = launches;
    return rc;
  }
  const Layout S = layout_saved(dims);
  // x in expert order comes from the forward (`saved`); dY is pulled here
  void* xs = at<void*>(const_cast<void*>(saved), S.off[SV_XS]);
  void* dys = at<void*>(ws, L.off[BW_DYS]);
  void* dG = at<void*>(ws, L.off[BW_DG]);
  void* dU = at<void*>(ws, L.off[BW_DU]);
  void* hw = at<void*>(ws, L.off[BW_HW]);
  void* dGsh = at<void*>(ws, L.off[BW_DGSH]);
  void* dUsh = at<void*>(ws, L.off[BW_DUSH]);
  void* hwsh = at<void*>(ws, L.off[BW_HWSH]);
  float* P = at<float*>(ws, L.off[BW_P]);
  void* dl = at<void*>(ws, L.off[BW_DL]);
  void* dXs = at<void*>(ws, L.off[BW_DXS]);
  void* dXsh = at<void*>(ws, L.off[BW_DXSH]);
  const int ldl = (E + 63) & ~63;
  const int grid_cap = num_sms();

  // 1. gather dY rows into each expert's region
  rc = cuda_status(launch_gather_rows("gather_dy", dY, nullptr, inv_pos, T, dims->k, 2 * d, dys, nullptr, s));
  if (rc != MOK_OK) return rc;
  ++launches;
  // 2. a = dY W_down^T; epilogue: dG, dU, w*h and the router partials <a, h>
  const int bn_da = bwd_bn_da(dims);
  {
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], dY, T, d, 64, 128);
      ok &= map3d(&p.maps[MS_B0], w->Ws_down, 1, Fs, d, 64, bn_da);
    }
    ok &= map2d(&p.maps[MS_A3], dys, R, d, 64, 128);
    ok &= map3d(&p.maps[MS_B3], w->W_down, E, F, d, 64, bn_da);
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = Fs / bn_da;
    p.nt[1] = F / bn_da;
    p.in0[0] = at<void*>(const_cast<void*>(saved), S.off[SV_GSH]);
    p.in1[0] = at<void*>(const_cast<void*>(saved), S.off[SV_USH]);
    p.in0[1] = at<void*>(const_cast<void*>(saved), S.off[SV_G]);
    p.in1[1] = at<void*>(const_cast<void*>(saved), S.off[SV_U]);
    p.out0[0] = dGsh; p.out1[0] = dUsh; p.out2[0] = hwsh;
    p.out0[1] = dG; p.out1[1] = dU; p.out2[1] = hw;
    p.row_w = sorted_w;
    p.partial = P;
    p.status = static_cast<int*>(ws);
    const int64_t bound = (sh ? (T + BM - 1) / BM * p.nt[0] : 0) + ((R + BM - 1) / BM + E) * p.nt[1];
    rc = cuda_status(launch_gemm(G_BWD_DA, bn_da, p, (int)std::min<int64_t>(grid_cap, bound), s));
    if (rc != MOK_OK) return rc;
    ++launches;
  }
  // 3. router backward: dw, dlogits, bf16 copy of dlogits
  rc = cuda_status(launch_router_backward(T, E, dims->k, F / bn_da, topk_idx, topk_w, inv_pos, P,
                                          dlogits, dl, s));
  if (rc != MOK_OK) return rc;
  ++launches;
  // 4. dX_s = dG W_gate^T + dU W_up^T; shared rows also take dl W_router^T
  {
    const int bn = bn_for(d, 256, 256);
    GemmParams p{};
    bool ok = true;
    int g0 = 0;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], dGsh, T, Fs, 64, 128);
      ok &= map3d(&p.maps[MS_B0], w->Ws_gate, 1, d, Fs, 64, bn);
      ok &= map2d(&p.maps[MS_A1], dUsh, T, Fs, 64, 128);
      ok &= map3d(&p.maps[MS_B1], w->Ws_up, 1, d, Fs, 64, bn);
      p.segkb[0][0] = Fs / BK;
      p.segkb[0][1] = Fs / BK;
      g0 = 2;
    }
    ok &= map2d(&p.maps[MS_A0 + g0], dl, T, ldl, 64, 128);
    ok &= map3d(&p.maps[MS_B0 + g0], w->W_router, 1, d, E, 64, bn);
    p.segkb[0][g0] = ldl / BK;
    ok &= map2d(&p.maps[MS_A3], dG, R, F, 64, 128);
    ok &= map3d(&p.maps[MS_B3], w->W_gate, E, d, F, 64, bn);
    ok &= map2d(&p.maps[MS_A4], dU, R, F, 64, 128);
    ok &= map3d(&p.maps[MS_B4], w->W_up, E, d, F, 64, bn);
    p.segkb[1][0] = F / BK;
    p.segkb[1][1] = F / BK;
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = 1;  // group 0 (shared expert and/or router term) always present
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.nt[0] = d / bn;
    p.nt[1] = d / bn;
    p.out0[0] = dXsh;
    p.out0[1] = dXs;
    p.status = static_cast<int*>(ws);
    const int64_t bound = (T + BM - 1) / BM * p.nt[0] + ((R + BM - 1) / BM + E) * p.nt[1];
    rc = cuda_status(launch_gemm(G_BWD_DX, bn, p, (int)std::min<int64_t>(grid_cap, bound), s));
    if (rc != MOK_OK) return rc;
    ++launches;
  }
  // 5. weight gradients (K = tokens of each expert, in token order) and x^T dl
  {
    const int bn = bn_for(d, F, sh ? Fs : 256);
    GemmParams p{};
    bool ok = true;
    if (sh) {
      ok &= map2d(&p.maps[MS_A0], x, T, d, 64, 64);
      ok &= map2d(&p.maps[MS_A1], hwsh, T, Fs, 64, 64);
      ok &= map2d(&p.maps[MS_B0], dGsh, T, Fs, 64, 64);
      ok &= map2d(&p.maps[MS_B1], dUsh, T, Fs, 64, 64);
      ok &= map2d(&p.maps[MS_B2], dY, T, d, 64, 64);
    }
    ok &= map2d(&p.maps[MS_A3], xs, R, d, 64, 64);
    ok &= map2d(&p.maps[MS_A4], hw, R, F, 64, 64);
    ok &= map2d(&p.maps[MS_B3], dG, R, F, 64, 64);
    ok &= map2d(&p.maps[MS_B4], dU, R, F, 64, 64);
    ok &= map2d(&p.maps[MS_B5], dys, R, d, 64, 64);
    if (dW_router) {
      ok &= map2d(&p.maps[MS_R_A], x, T, d, 64, 64);
      ok &= map2d(&p.maps[MS_R_B], dl, T, ldl, 64, 64);
      p.router_tiles = (d / BM) * ((E + bn - 1) / bn);
      p.E_cols = E;
      p.out_router = dW_router;
    }
    if (!ok) return MOK_ERR_CUDA;
    p.offsets = offsets;
    p.E = E;
    p.has_shared = sh;
    p.T = (int)T;
    p.d = d;
    p.F = F;
    p.Fs = Fs;
    p.out0[0] = dWs_gate; p.out1[0] = dWs_up; p.out2[0] = dWs_down;
    p.out0[1] = dW_gate; p.out1[1] = dW_up; p.out2[1] = dW_down;
    // the routed operands' maps bounded to each expert's rows
    CUtensorMap* emaps = at<CUtensorMap*>(ws, L.off[BW_TMAP]);
    {
      BoundMapParams bp{};
      const int slot[kBoundMaps] = {MS_A3, MS_A4, MS_B3, MS_B4, MS_B5};
      const void* base[kBoundMaps] = {xs, hw, dG, dU, dys};
      const int cols[kBoundMaps] = {d, F, F, F, d};
      for (int j = 0; j < kBoundMaps; ++j) {
        bp.templ[j] = p.maps[slot[j]];
        bp.base[j] = base[j];
        bp.cols[j] = cols[j];
      }
      bp.offsets = offsets;
      bp.E = E;
      bp.emaps = emaps;
      rc = cuda_status(launch_dw_bound_maps(bp, s));
      if (rc != MOK_OK) return rc;
      ++launches;
    }
    p.emaps = emaps;
    p.status = static_cast<int*>(ws);
    const int64_t total = p.router_tiles +
                          (sh ? 2 * (d / BM) * (Fs / bn) + (Fs / BM) * (d / bn) : 0) +
                          (int64_t)E * (2 * (d / BM) * (F / bn) + (F / BM) * (d / bn));
    // CTA pairs (adjacent M tiles of one problem; each SM stages half the B columns) when every
    // problem's M-tile count is even
    const bool dw_pair = bn == 256 && (d / BM) % 2 == 0 && (F / BM) % 2 == 0 && (!sh || (Fs / BM) % 2 == 0);
    rc = cuda_status(launch_gemm(G_BWD_DW, bn, p, (int)std::min<int64_t>(grid_cap, total), s, dw_pair));
    if (rc != MOK_OK) return rc;
    ++launches;
  }
  // 6. dX = dX_shared (+ router term) + routed rows in ascending expert order
  rc = cuda_status(launch_combine(T, d, dims->k, topk_idx, inv_pos, dXs, dXsh, dX, s));
  if (rc != MOK_OK) return rc;
  ++launches;
  g_last_launches = launches;
  return MOK_OK;
}

}  // extern "C"

// Per-workspace state of the host entry point: which of its two device x buffers the next call
// fills, and per buffer the event of its copy landing and of the layer being done reading it.
// A small table keyed by (device, workspace); its oldest entry is reused (after waiting for its
// events) when a new workspace comes.
struct HostPipe {
  const void* ws = nullptr;
  int device = -1;
  cudaEvent_t ready[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
  int next = 0;
  uint64_t last_use = 0;
};
constexpr int kHostPipes = 16;
static std::mutex g_pipe_mu;
static HostPipe g_pipes[kHostPipes];
static uint64_t g_pipe_clock = 0;
constexpr int kMaxDevices = 64;
static cudaStream_t g_copy_stream[kMaxDevices] = {};

static cudaError_t host_pipe(const void* ws, HostPipe** out, cudaStream_t* copy) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  if (!g_copy_stream[dev]) {
    e = cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *copy = g_copy_stream[dev];
  HostPipe* hit = nullptr;
  HostPipe* oldest = &g_pipes[0];
  for (HostPipe& P : g_pipes) {
    if (P.ws == ws && P.device == dev) hit = &P;
    if (P.last_use < oldest->last_use) oldest = &P;
  }
  if (!hit) {
    hit = oldest;
    if (hit->ready[0]) {  // reused: its previous workspace's copies and readers are done first
      for (int b = 0; b < 2; ++b) {
        if ((e = cudaEventSynchronize(hit->ready[b])) != cudaSuccess) return e;
        if ((e = cudaEventSynchronize(hit->freed[b])) != cudaSuccess) return e;
      }
      if (hit->device != dev) {
        for (int b = 0; b < 2; ++b) {
          cudaEventDestroy(hit->ready[b]);
          cudaEventDestroy(hit->freed[b]);
          hit->ready[b] = hit->freed[b] = nullptr;
        }
      }
    }
    if (!hit->ready[0]) {
      for (int b = 0; b < 2; ++b) {
        if ((e = cudaEventCreateWithFlags(&hit->ready[b], cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&hit->freed[b], cudaEventDisableTiming)) != cudaSuccess) return e;
      }
    }
    hit->ws = ws;
    hit->device = dev;
    hit->next = 0;
  }
  hit->last_use = ++g_pipe_clock;
  *out = hit;
  return cudaSuccess;
}

extern "C" {

int mok_layer_forward_host(const mok_dims* dims, const mok_weights* w, const void* x_host,
                           void* y_host, void* ws, size_t ws_bytes, mok_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != MOK_OK) return rc;
  if (!w || !ws || !x_host || !y_host) return MOK_ERR_INVALID_ARG;
  const size_t fw = layout_fwd(dims).total;
  const Layout H = layout_host(dims);
  if (ws_bytes < fw + H.total) return MOK_ERR_WORKSPACE;
  if (dims->T == 0) return MOK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ext = static_cast<char*>(ws) + fw;
  const size_t xbytes = 2ull * dims->T * dims->d;
  HostPipe* P = nullptr;
  cudaStream_t copy = nullptr;
  if (host_pipe(ws, &P, &copy) != cudaSuccess) return MOK_ERR_CUDA;
  const int b = P->next;
  P->next ^= 1;
  void* x = ext + H.off[HS_X] + b * al(xbytes);
  void* y = ext + H.off[HS_Y];
  int32_t* idx = reinterpret_cast<int32_t*>(ext + H.off[HS_IDX]);
  float* tw = reinterpret_cast<float*>(ext + H.off[HS_W]);
  int32_t* cnt = reinterpret_cast<int32_t*>(ext + H.off[HS_CNT]);
  int32_t* off = reinterpret_cast<int32_t*>(ext + H.off[HS_OFF]);
  int32_t* stok = reinterpret_cast<int32_t*>(ext + H.off[HS_STOK]);
  float* sw = reinterpret_cast<float*>(ext + H.off[HS_SW]);
  int32_t* inv = reinterpret_cast<int32_t*>(ext + H.off[HS_INV]);
  // the copy waits until the call two back (same buffer) is done reading it; the layer waits
  // for the copy
  if (cudaStreamWaitEvent(copy, P->freed[b], 0) != cudaSuccess) return MOK_ERR_CUDA;
  if (cudaMemcpyAsync(x, x_host, xbytes, cudaMemcpyHostToDevice, copy) != cudaSuccess) return MOK_ERR_CUDA;
  if (cudaEventRecord(P->ready[b], copy) != cudaSuccess) return MOK_ERR_CUDA;
  if (cudaStreamWaitEvent(s, P->ready[b], 0) != cudaSuccess) return MOK_ERR_CUDA;
  int total = 0;
  rc = mok_route(dims, x, w->W_router, w->router_bias, idx, tw, nullptr, ws, fw, stream);
  if (rc != MOK_OK) return rc;
  total += g_last_launches;
  rc = mok_dispatch_index(dims, idx, tw, cnt, off, stok, sw, inv, ws, fw, stream);
  if (rc != MOK_OK) return rc;
  total += g_last_launches;
  // pinned (mapped) y_host: the combine writes y straight into host memory; otherwise y is
  // combined in the workspace and copied back
  cudaPointerAttributes ya{};
  void* y_out = y;
  if (cudaPointerGetAttributes(&ya, y_host) == cudaSuccess && ya.type == cudaMemoryTypeHost &&
      ya.devicePointer && aligned16(ya.devicePointer))
    y_out = ya.devicePointer;
  else
    cudaGetLastError();  // pageable memory: not an error for this call
  rc = mok_moe_forward(dims, w, x, idx, off, stok, sw, inv, y_out, nullptr, ws, fw, stream);
  if (rc != MOK_OK) return rc;
  total += g_last_launches;
  if (cudaEventRecord(P->freed[b], s) != cudaSuccess) return MOK_ERR_CUDA;
  if (y_out == y &&
      cudaMemcpyAsync(y_host, y, xbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOK_ERR_CUDA;
  g_last_launches = total;
  return MOK_OK;
}

}  // extern "C"
