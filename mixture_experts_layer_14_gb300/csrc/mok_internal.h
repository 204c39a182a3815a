// Internal declarations shared by the host code and the kernels of libmok.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mok.h"

namespace mok {

constexpr uint64_t kWaitNs = 2000000000ull;  // bounded device waits give up after 2 s
constexpr int BM = 128;                      // UMMA M: rows of a tile (TMEM lanes)
constexpr int BK = 64;                       // K per pipeline stage: 64 bf16 = one 128 B row
constexpr int kGemmThreads = 192;            // warp 0 TMA, warp 1 MMA/TMEM, warps 2..5 epilogue
constexpr int kDispatchChunk = 64;           // tokens per histogram block of the counting sort
constexpr int kMaxE = 512;
// NVFP4 GEMMs: A tiles of at most this many rows are loaded through 32-row-box maps (MS_A1 for
// the shared expert, MS_A4 for the routed experts)
constexpr int kNvSmallRows = 32;
constexpr int kMaxK = 8;
constexpr int kBoundMaps = 5;                   // G_BWD_DW: expert-bounded maps per expert

// ------------------------------------------------------------------ grouped GEMM
enum GemmMode : int {
  G_FWD_GU = 0,    // h = SiLU(X Wg) * (X Wu)              M-grouped, A K-major, B MN-major
  G_FWD_DOWN = 1,  // Y = w * (h Wd)                       M-grouped, A K-major, B MN-major
  G_BWD_DA = 2,    // a = dY Wd^T -> dG, dU, w*h, <a,h>    M-grouped, A K-major, B K-major
  G_BWD_DX = 3,    // dX = dG Wg^T + dU Wu^T (+ dl Wr^T)   M-grouped, A K-major, B K-major
  G_BWD_DW = 4,    // dW = X^T dG, X^T dU, (w h)^T dY, x^T dl  K-grouped, A and B MN-major
  G_FWD_GU_MX = 5,   // MXFP8 gate/up: h quantised to E4M3 + UE8M0 in the epilogue
  G_FWD_DOWN_MX = 6, // MXFP8 down: Y = w * (h Wd), bf16 out
  // MXFP8 backward (every operand E4M3 + UE8M0 along the GEMM's own K, both K-major):
  G_BWD_DA_MX = 7,   // a = dY Wd^T -> dG, dU along F; dG, dU, w*h along tokens; <a,h>
  G_BWD_DX_MX = 8,   // dX = dG Wg^T + dU Wu^T                      M-grouped
  G_BWD_DW_MX = 9,   // dW from operands quantised along tokens     K-grouped (transposed)
  // gate/up + SwiGLU, then down + router weight, in one persistent launch: CTAs claim tiles from
  // a device work counter (every gate/up tile before any down tile), and a down tile waits for
  // the readiness counter of its M tile (all its h columns written)
  G_FWD_GUD = 10,
  // NVFP4 (f16 operands on the tensor cores): A = activations holding NVFP4 values (q * s), B =
  // NVFP4 weight codes and block scales decoded into f16 in shared memory by converter warps;
  // the tensor scales are applied in the epilogue
  G_FWD_GU_NV = 11,   // h = SiLU(X Wg) * (X Wu), quantised to NVFP4 values (f16) in the epilogue
  G_FWD_DOWN_NV = 12, // Y = w * (h Wd), bf16 out
};

// Tensor-map slots.  Group 0 is the shared expert (rows = tokens), group 1 the routed experts
// (rows = destination rows of the pull schedule).  Which slots a mode uses is listed in
// moe_gemm.cu next to its producer.
enum MapSlot : int {
  MS_A0 = 0, MS_A1 = 1, MS_A2 = 2,  // group 0 A operands (per segment / sub-GEMM)
  MS_A3 = 3, MS_A4 = 4, MS_A5 = 5,  // group 1 A operands
  MS_B0 = 6, MS_B1 = 7, MS_B2 = 8,  // group 0 B operands
  MS_B3 = 9, MS_B4 = 10, MS_B5 = 11,  // group 1 B operands
  MS_R_A = 12, MS_R_B = 13,           // router GEMM of the backward (x^T dl)
  MS_COUNT = 14
};

struct GemmParams {
  CUtensorMap maps[MS_COUNT];
  const int* offsets;   // routed row offsets [E+1] (device), NULL when E == 0
  int E;                // routed experts in this launch (0 = none)
  int has_shared;       // group 0 present
  int T;                // rows of group 0
  int d, F, Fs;         // layer dims
  int nt[2];            // N tiles per group (M-grouped modes)
  int nseg[2];          // K segments per group (G_BWD_DX)
  int segkb[2][3];      // k-blocks of each segment
  int router_tiles;     // G_BWD_DW: number of x^T dl tiles (0 = none)
  int E_cols;           // G_BWD_DW: valid columns of dW_router (= E)
  // epilogue pointers, [group]
  void* out0[2];        // h / Y / dG / dX / dW_gate
  void* out1[2];        // G (saved)      / dU / dW_up
  void* out2[2];        // U (saved)      / w*h / dW_down; G_FWD_GU_MX: G (saved, fp32) or NULL
  void* out3[2];        // G_FWD_GU_MX: U (saved, fp32) or NULL
  void* out_router;     // dW_router [d,E]
  const void* in0[2];   // G (saved) for G_BWD_DA (bf16) and G_BWD_DA_MX (fp32)
  const void* in1[2];   // U (saved)
  const float* row_w;   // router weight of each routed row (sorted_w)
  float* partial;       // G_BWD_DA: <a,h> per (routed row, N tile), [R, nt[1]]
  // MXFP8 scale factors as scale atoms (mok_mx.cuh), [group]: A by M tile (the tile's index in
  // the M-grouped decode), B by 128-row tile of each expert's K-major weight; the weight-gradient
  // GEMM's transposed operands by 128-row tile and K block of the whole matrix.
  //  gate/up: sfa x; sfb gate, up.  down: sfa h; sfb down.  da: sfa dY; sfb down.
  //  dx: sfa dG, dU; sfb gate, up.  dw: sfa x^T, (w h)^T; sfb dG^T, dU^T, dY^T.
  const uint8_t* sfa[2][2];
  const uint8_t* sfb[2][3];
  int sf_kb[2];                // K blocks of 128 per row of the scale atoms
  // G_BWD_DA_MX: E4M3 codes [rows][F] and scale atoms (by M tile) of dG and dU, [group][dG, dU]
  void* qout[2][2];
  uint8_t* qsc[2][2];
  // G_BWD_DA_MX: dG, dU and w*h quantised along tokens for the weight gradients, transposed:
  // codes [F][128 tnkb] (the M tile mt's rows are columns 128 mt ..), atoms [F/128][tnkb]
  uint8_t* tq[2][3];
  uint8_t* tsc[2][3];
  int tnkb[2];
  // G_BWD_DW: per expert, kBoundMaps copies of the routed operands' maps bounded to its rows
  // (x_sorted, w*h, dG, dU, dY_sorted), from launch_dw_bound_maps
  const CUtensorMap* emaps;
  // G_FWD_GUD: N tiles of the down phase per group; the work counter (work[0], zero at launch)
  // and one readiness counter per M tile (shared expert's first, zero at launch)
  int ntb[2];
  int* work;
  int* ready;
  int nfast_mt;         // M-grouped: groups of at least this many M tiles run N tiles fastest (0: never)
  // K-grouped tile decode: the launch's runtime divisors as m = ceil(2^32 / divisor), so that
  // n / divisor = (n * m) >> 32 (exact for n * divisor < 2^32, checked at launch): tiles per
  // routed problem, N tiles per row of a gate/up gradient [group], of a down gradient, and of
  // the router gradient (router_nt of them)
  uint64_t dm_per, dm_nt[2], dm_ntd, dm_ntr;
  int router_nt;
  // NVFP4 modes, [group][gate or down, up]: weight code rows (32 bytes) and scale rows (4 bytes)
  // per (expert, 64-element K block, N row), the per-expert decode scales 1 / S, and the
  // calibrated activation amaxes {x, h}
  const uint8_t* nvq[2][2];
  const uint8_t* nvs[2][2];
  const float* nvg[2][2];
  const float* nv_act;
  int* status;
};

// Expert-bounded copies of the weight-gradient GEMM's routed operand maps (moe_gemm.cu):
// templ[j] over the whole tensor base[j] (row-major, cols[j] bf16 per row), for j = x_sorted,
// w*h, dG, dU, dY_sorted; emaps[e * kBoundMaps + j] gets the copy bounded to expert e's rows.
struct BoundMapParams {
  CUtensorMap templ[kBoundMaps];
  const void* base[kBoundMaps];
  int cols[kBoundMaps];
  const int* offsets;
  int E;
  CUtensorMap* emaps;
};
cudaError_t launch_dw_bound_maps(const BoundMapParams& bp, cudaStream_t s);

// Launches (moe_gemm.cu).  grid = persistent CTAs.
// pair: bf16 gate/up and down (N tile 256) in CTA pairs of 256-row tiles, or the weight-gradient
// GEMM in pairs of adjacent M tiles (cluster launch).
cudaError_t launch_gemm(int mode, int bn, const GemmParams& p, int grid, cudaStream_t s,
                        bool pair = false);

// Router (route.cu)
struct RouteParams {
  CUtensorMap map_x;   // x [T,d] K-major, box {64,128}
  CUtensorMap map_w;   // W_router [d,E] MN-major, box {64,64}
  const float* bias;
  int32_t* topk_idx;
  float* topk_w;
  float* logits;
  int T, d, E, k;
  int splits;          // K splits per 128-token tile: a cluster of `splits` CTAs (power of two)
  int chunk;           // splits > 1: logit columns reduced through shared memory per pass
  int* status;
};
constexpr int kMaxRouteSplits = 8;
int route_splits(int64_t T, int d);
cudaError_t launch_route(const RouteParams& p, cudaStream_t s);

// Dispatch (dispatch.cu)
cudaError_t launch_dispatch(int64_t T, int E, int k, const int32_t* topk_idx, const float* topk_w,
                            int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                            float* sorted_w, int32_t* inv_pos, int32_t* hist, int* status,
                            cudaStream_t s, int* launches);

// Elementwise (elementwise.cu)
// Row gathers: dst[r] = src[rows[r]] for r < nrows; an index outside [0, nsrc) gives a zero row.
// Token-major pull gather: dst[inv_pos[t, j]] = src[t] for every kept route (rows of row_bytes,
// a multiple of 16); a second source / destination pair (or NULL) moves the same way.
cudaError_t launch_gather_rows(const char* name, const void* src0, const void* src1,
                               const int32_t* inv_pos, int64_t T, int k, int row_bytes,
                               void* dst0, void* dst1, cudaStream_t s);
// y[t] = Ysh[t] (+ Ysh2[t]) + routed rows in ascending expert order; Ysh, Ysh2 may be NULL.
cudaError_t launch_combine(int64_t T, int d, int k, const int32_t* topk_idx,
                           const int32_t* inv_pos, const void* Ys, const void* Ysh, void* y,
                           cudaStream_t s, const void* Ysh2 = nullptr);
cudaError_t launch_router_backward(int64_t T, int E, int k, int ldp, const int32_t* topk_idx,
                                   const float* topk_w, const int32_t* inv_pos,
                                   const float* partial, float* dlogits, void* dl_bf16,
                                   cudaStream_t s);

int num_sms();

// MXFP8 quantisation (mx.cu); scale atoms are described in mok_mx.cuh
cudaError_t launch_mx_quantize_rows(const void* src, int64_t rows, int K, void* q, void* sc,
                                    bool atoms, cudaStream_t s);
cudaError_t launch_gather_scale_atoms(const void* src, const int32_t* sorted_tok,
                                      const int32_t* offsets, int E, int64_t T, int64_t R, int K,
                                      void* dst, cudaStream_t s);
cudaError_t launch_mx_quantize_transpose(const void* src, int64_t nmat, int K, int N, void* q,
                                         void* sc, cudaStream_t s);
// MXFP8 backward: rows of each expert (src rows rows_idx[offsets[e] + i], or offsets[e] + i
// without rows_idx; one segment of nsrc rows when offsets is NULL) quantised along tokens into
// the transposed codes q[C][128 nkb] (expert e at columns 128 s_mt[e], zero-padded to whole
// 128-column blocks) and scale atoms [C/128][nkb]; up to three operands of the same rows and
// width C (a multiple of 64) per launch.
struct TokQuantParams {
  const __nv_bfloat16* src[3];
  uint8_t* q[3];
  uint8_t* sc[3];
  int nops;
  int C;
  int64_t nsrc;
  const int32_t* rows_idx;
  const int32_t* offsets;
  int E;
  int nkb;
};
cudaError_t launch_mx_quantize_tokens(const TokQuantParams& tp, cudaStream_t s);
// NVFP4 quantisation (nv.cu; format and recipe in mok_nv.cuh).  launch_nv_prepare: per-matrix
// amax (amax[m] must be zero at launch) then codes and block scales of src [nmat][K][N] as rows
// of 32 + 4 bytes per (matrix, 64-element K block, column) and g[m] = 1 / S.
// launch_nv_quantize_act: rows x K bf16 -> f16 NVFP4 values without the tensor scale, with the
// calibrated tensor amax *amax.
cudaError_t launch_nv_prepare(const void* src, int64_t nmat, int K, int N, uint32_t* amax, void* q,
                              void* sc, float* g, cudaStream_t s);
cudaError_t launch_nv_quantize_act(const void* src, int64_t rows, int K, const float* amax,
                                   void* dst, cudaStream_t s);
cudaError_t launch_nv_set_act(float* act, float amax_x, float amax_h, cudaStream_t s);
// Optional per-launch CUDA-event timing (profile.cu); no-ops unless enabled on this thread.
void prof_begin(const char* name, cudaStream_t s);
void prof_end(cudaStream_t s);

}  // namespace mok
