/*
 * mok.h — C ABI of the GB300 (sm_103a) DeepSeek-V3-style mixture-of-experts layer.
 *
 * The layer (page "Mixture-of-Kittens: Nhân kernel MoE nguồn mở tối ưu cho hệ thống NVL72",
 * section "Chồng lấp tính toán và truyền tải trong MoE"): a router projection picks the top-k
 * routed experts of every token and gives each a router weight; every selected expert runs a
 * SwiGLU FFN (gate and up projections, SiLU(gate) * up, down projection); the output is the
 * always-on shared expert plus the router-weighted sum of the routed experts:
 *
 *     logits = x W_router + b                     (fp32)
 *     topk   = the k largest logits, ties to the lower expert index
 *     w_j    = softmax(logits)[e_j] / sum_{i<k} softmax(logits)[e_i]
 *     y      = FFN_shared(x) + sum_j w_j FFN_{e_j}(x),   FFN(x) = (SiLU(x Wg) * (x Wu)) Wd
 *
 * Dispatch follows the pull schedule of the same page, section "Lập lịch" (each expert's
 * destination rows list its source tokens; one GPU, so the source rank is always 0) and the
 * pull example of the page "Метод и эксперименты" (tokens ascend inside an expert's region).
 * Results are bit-identical from run to run (page "Mixture-of-Kittens; MoE megakernel", key
 * points): every reduction runs in a fixed order and no floating-point atomics are used.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *    The library never allocates, frees or synchronises (except mok_read_device_status and the
 *    host-buffer entry point, which say so).  Work is enqueued on `stream` and runs
 *    asynchronously.
 *  - Layouts are row-major and dense: x[T,d], W_router[d,E], W_gate/W_up[E,d,F],
 *    W_down[E,F,d], Ws_gate/Ws_up[d,Fs], Ws_down[Fs,d]; bf16 unless noted.
 *  - Preconditions (checked on the host; violations return MOK_ERR_UNSUPPORTED or
 *    MOK_ERR_INVALID_ARG and enqueue nothing): T >= 0; d % 128 == 0; F % 128 == 0;
 *    Fs % 128 == 0 when n_shared == 1; n_shared in {0,1}; 1 <= k <= 8; k <= E <= 512;
 *    E % 8 == 0; every pointer 16-byte aligned; workspace at least mok_workspace_size().
 *  - Device-side failures (a bounded wait that ran out, an out-of-range expert index) are
 *    recorded as a nonzero status word inside the workspace; nothing traps.  Read it with
 *    mok_read_device_status().  The word is sticky: clear it with mok_clear_device_status()
 *    (or allocate the workspace zeroed).
 *  - Return value: MOK_OK or a negative mok_status.  No entry point exits or aborts.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mok_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad enum */
  MOK_ERR_UNSUPPORTED = -2, /* shape or alignment outside the preconditions */
  MOK_ERR_WORKSPACE = -3,   /* workspace too small */
  MOK_ERR_CUDA = -4,        /* a CUDA runtime / driver call failed */
  MOK_ERR_TIMEOUT = -5,     /* (device status) a bounded wait inside a kernel ran out */
  MOK_ERR_DEVICE_CHECK = -6 /* (device status) an index failed a device-side range check */
} mok_status;

typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1, MOK_NVFP4 = 2 } mok_dtype;

typedef enum { MOK_PASS_FORWARD = 0, MOK_PASS_BACKWARD = 1 } mok_pass;

/* Sizes of one layer call.  T tokens, d model dim, E routed experts, k experts per token,
 * F routed-expert intermediate, F_shared shared-expert intermediate, n_shared in {0,1},
 * dtype = arithmetic of the expert GEMMs (MOK_MXFP8: E4M3 values with one UE8M0 scale per
 * 32 elements along the reduction dimension; MOK_NVFP4: E2M1 values with one E4M3 scale per
 * 16 elements along the reduction dimension and one fp32 scale per tensor, forward only; the
 * router and combine stay fp32/bf16). */
typedef struct {
  int64_t T;
  int32_t d, E, k, F, F_shared, n_shared;
  int32_t dtype;
} mok_dims;

/* Layer weights (device, caller-owned). `prepared` is the output of mok_prepare_weights and is
 * required when dtype is MOK_MXFP8 or MOK_NVFP4 (ignored for MOK_BF16); `prepared_bwd`, the output of
 * mok_prepare_weights_bwd, is required by mok_moe_backward when dtype == MOK_MXFP8. */
typedef struct {
  const void *W_router;     /* [d,E] bf16 */
  const float *router_bias; /* [E] fp32, or NULL */
  const void *W_gate;       /* [E,d,F] bf16 */
  const void *W_up;         /* [E,d,F] bf16 */
  const void *W_down;       /* [E,F,d] bf16 */
  const void *Ws_gate;      /* [d,Fs] bf16 (NULL when n_shared == 0) */
  const void *Ws_up;        /* [d,Fs] bf16 */
  const void *Ws_down;      /* [Fs,d] bf16 */
  const void *prepared;     /* mok_prepared_size() bytes, or NULL */
  const void *prepared_bwd; /* mok_prepared_bwd_size() bytes, or NULL */
} mok_weights;

/* Bytes of device workspace needed by the entry points of `pass` (MOK_PASS_FORWARD covers
 * mok_route, mok_dispatch_index and mok_moe_forward; MOK_PASS_BACKWARD covers
 * mok_moe_backward).  Returns 0 for invalid dims. */
size_t mok_workspace_size(const mok_dims *dims, int pass);

/* Bytes of the activations mok_moe_forward saves for mok_moe_backward: G and U for the routed
 * rows and the shared expert (bf16 for MOK_BF16, fp32 for MOK_MXFP8, whose backward quantises
 * dG, dU and w*h derived from them), and with MOK_BF16 also x in expert order. */
size_t mok_saved_size(const mok_dims *dims);

/* Bytes of the prepared-weights buffer for dims->dtype (0 for MOK_BF16). */
size_t mok_prepared_size(const mok_dims *dims);

/* MXFP8: quantise the routed and shared expert weights once into `prepared` (E4M3 values and
 * UE8M0 scales, blocks of 32 along each weight's reduction dimension, same rule as
 * mok_mx_quantize_rows), transposed to K-major, in this order (each region 1 KB aligned):
 * W_gate codes [E][F][d] and scales; W_up likewise; W_down codes [E][d][F] and scales; then the
 * shared expert's three the same way.  The scales of a K-major matrix [N][K] (N rows, K/32 scale
 * bytes per row) are stored in 512-byte atoms [N/128][K/128]: the atom of row tile a and K block
 * b holds row n = 128a + 32 r1 + r0 (r0 < 32, r1 < 4), block 4b + j at byte 16 r0 + 4 r1 + j,
 * the shared-memory image the block-scaled MMA's scale copy reads.  No-op for MOK_BF16.
 * MXFP8 needs d % 256 == 0. */
int mok_prepare_weights(const mok_dims *dims, const mok_weights *w, void *prepared,
                        mok_stream_t stream);
/* NVFP4 (MOK_NVFP4; the first page, "Mixture-of-Kittens: Nhân kernel MoE ...", names NVFP4 as
 * the format of its authors' earlier kernels and defines neither format nor recipe; the format
 * is NVIDIA's NVFP4 and the recipe the plain two-level one): mok_prepare_weights quantises every
 * expert weight along its reduction dimension (K = d for gate and up, F for down), each matrix
 * with its own tensor scale: A = the matrix's amax, S = 2688 / A in fp32 (1 when A is 0); a block
 * of 16 with amax a takes the E4M3 scale s = rn((a / 6) * S) (saturating); an element v the E2M1
 * code rn(v * (S / s)) (ties to the even code, saturating at 6; sign bit when the product is
 * negative; 0 when s is 0); every step an fp32 operation rounded to nearest even.  Layout, in
 * this order, each region 1 KB aligned: W_gate codes, W_gate scales, W_up codes, W_up scales,
 * W_down codes, W_down scales, the shared expert's six likewise (E = 1), then g[3E + 3] fp32
 * (1 / S of gate e, up e, down e for e < E, then the shared gate, up, down), amax[3E + 3]
 * (scratch), act[2] fp32 (the calibrated activation amaxes, below).  Codes of a matrix with K
 * rows and N columns: for each 64-element K block kb and column n, 32 bytes at
 * ((m * K/64 + kb) * N + n) * 32 (m = the expert), byte j holding elements 2j (low nibble) and
 * 2j + 1 (high nibble) of the block; its 4 scale bytes (one per 16 elements) at
 * ((m * K/64 + kb) * N + n) * 4.  The activation amaxes are reset to 0 (tensor scale 1).
 * NVFP4 needs d % 256 == 0. */

/* NVFP4: sets the calibrated tensor amaxes of the forward's two quantised activations, x (the
 * layer input, quantised along d) and h (SiLU(G) * U, quantised along F from its fp32 value),
 * in `prepared` (the static form of the per-tensor scale: values beyond them saturate).  Both
 * must be finite and >= 0 (0 gives the tensor scale 1).  Returns MOK_ERR_INVALID_ARG for another
 * dtype, a NULL or unaligned buffer, or a negative or non-finite amax. */
int mok_nvfp4_set_activation_amax(const mok_dims *dims, void *prepared, float amax_x,
                                  float amax_h, mok_stream_t stream);

/* MXFP8 backward: the expert weights quantised once more, along the reduction dimension of the
 * backward GEMM that reads each (same rule and atom layout as mok_prepare_weights), in this order
 * (each region 1 KB aligned): W_down codes [E][F][d] (blocks along d, for dY W_down^T) and
 * scales; W_gate codes [E][d][F] (blocks along F, for dG W_gate^T) and scales; W_up likewise;
 * then the shared expert's Ws_down [Fs][d], Ws_gate [d][Fs], Ws_up [d][Fs] the same way.  No
 * transposes: each weight's rows are already along that K.  mok_prepared_bwd_size() bytes
 * (0 for MOK_BF16, where this call is a no-op).  The MXFP8 backward needs F % 256 == 0 and
 * Fs % 256 == 0 besides d % 256 == 0. */
size_t mok_prepared_bwd_size(const mok_dims *dims);
int mok_prepare_weights_bwd(const mok_dims *dims, const mok_weights *w, void *prepared_bwd,
                            mok_stream_t stream);

/* MXFP8 quantiser of activations: src[rows,K] bf16 -> q[rows,K] E4M3 codes and
 * scales[rows,K/32] UE8M0 bytes, one block per 32 consecutive elements of a row: scale 2^s with
 * s the smallest integer such that amax <= 448 * 2^s (amax / 448 rounded up to a power of two),
 * s in [-127,127] (an all-zero block gets 0x00), codes = round-to-nearest-even E4M3 of v * 2^-s
 * with saturation to +-448.  K % 128 == 0.  The MXFP8 format of the layer (page
 * "Mixture-of-Kittens; MoE megakernel", key points); the scale rule as read for the MXFP8
 * workload of the layer. */
int mok_mx_quantize_rows(int64_t rows, int K, const void *src, void *q, void *scales,
                         mok_stream_t stream);

/* Router: logits = x W_router + bias in fp32 (bf16 tensor-core products, fp32 accumulation),
 * top-k by (logit descending, index ascending), weights = softmax over all experts
 * renormalised over the selected ones.  Page "Mixture-of-Kittens: Nhân kernel MoE ...",
 * section "Chồng lấp tính toán và truyền tải trong MoE".
 *   x[T,d] bf16, W_router[d,E] bf16, bias[E] fp32 or NULL
 *   -> topk_idx[T,k] int32 (slot order = descending logit), topk_w[T,k] fp32,
 *      logits[T,E] fp32 (optional, NULL to skip). */
int mok_route(const mok_dims *dims, const void *x, const void *W_router, const float *bias,
              int32_t *topk_idx, float *topk_w, float *logits, void *ws, size_t ws_bytes,
              mok_stream_t stream);

/* Pull schedule (page "Mixture-of-Kittens: Nhân kernel MoE ...", section "Lập lịch"): a
 * deterministic counting sort of the T*k routes by expert, built from per-chunk histograms and
 * a prefix scan, with no atomics.  Within an expert, routes are ordered by token id.
 *   topk_idx[T,k] int32 (each value in [0,E)), topk_w[T,k] fp32
 *   -> counts[E], offsets[E+1] (offsets[0]=0, offsets[E]=T*k), sorted_tok[T*k] (token of each
 *      destination row), sorted_w[T*k] (its router weight), inv_pos[T,k] (destination row of
 *      route (t,j)).  An index outside [0,E) sets MOK_ERR_DEVICE_CHECK in the status word and
 *      that route is dropped. */
int mok_dispatch_index(const mok_dims *dims, const int32_t *topk_idx, const float *topk_w,
                       int32_t *counts, int32_t *offsets, int32_t *sorted_tok, float *sorted_w,
                       int32_t *inv_pos, void *ws, size_t ws_bytes, mok_stream_t stream);

/* Forward of the expert part given a routing (the output of mok_dispatch_index):
 * pull-gathers each expert's rows, runs the gate/up GEMM with SiLU(gate)*up fused in its
 * epilogue and the down GEMM with the router weight fused in its epilogue (routed experts and
 * the shared expert in one persistent launch per phase), then combines every token's rows in
 * ascending expert order on top of the shared-expert row (fp32 accumulation, one bf16
 * rounding).
 *   -> y[T,d] bf16.  `saved` (mok_saved_size bytes or NULL) receives what the backward needs:
 *   G and U (bf16; for MOK_MXFP8 the block-scaled products in fp32), and for MOK_BF16 x in
 *   expert order.  MOK_NVFP4: x is quantised with its calibrated amax, the gate/up GEMM's
 *   epilogue quantises h along F, both GEMMs multiply f16 NVFP4 values decoded from the
 *   prepared weights and apply the tensor scales in their epilogues; forward only (`saved` must
 *   be NULL, else MOK_ERR_UNSUPPORTED). */
int mok_moe_forward(const mok_dims *dims, const mok_weights *w, const void *x,
                    const int32_t *topk_idx, const int32_t *offsets, const int32_t *sorted_tok,
                    const float *sorted_w, const int32_t *inv_pos, void *y, void *saved,
                    void *ws, size_t ws_bytes, mok_stream_t stream);

/* Backward of the layer for upstream gradient dY[T,d] bf16, with the top-k selection held
 * constant (unselected experts get no gradient).  Uses `saved` from mok_moe_forward with the
 * same routing.  Outputs (bf16 unless noted; fp32 accumulation, fixed summation order):
 *   dX[T,d] (including the router path dlogits W_router^T), dW_gate/dW_up[E,d,F],
 *   dW_down[E,F,d] (experts with no token get zeros), dWs_gate/dWs_up[d,Fs], dWs_down[Fs,d]
 *   (NULL when n_shared == 0), dlogits[T,E] fp32 (zero off the selection),
 *   dW_router[d,E] (NULL to skip).
 * MOK_MXFP8 (the MXFP8 reading of the training step): every expert GEMM multiplies E4M3
 * operands with UE8M0 scales per 32 along its own reduction dimension — dY and W_down along d,
 * dG, dU, W_gate, W_up along F, and for the weight gradients x, dG, dU, w*h and dY along each
 * expert's tokens (blocks of 32 from its first token, in token order) — with fp32 accumulation;
 * the router terms dlogits W_router^T and x^T dlogits stay bf16.  Needs w->prepared_bwd and a
 * `saved` from an MXFP8 forward; F % 256 == 0, Fs % 256 == 0 and
 * 2 (ceil(T k / 128) + E) d / 64 < 2^31 (T below about 150M tokens at d = 7168, k = 8), else
 * MOK_ERR_UNSUPPORTED.  MOK_NVFP4 has no backward: MOK_ERR_UNSUPPORTED. */
int mok_moe_backward(const mok_dims *dims, const mok_weights *w, const void *x, const void *dY,
                     const void *saved, const int32_t *topk_idx, const float *topk_w,
                     const int32_t *offsets, const int32_t *sorted_tok, const float *sorted_w,
                     const int32_t *inv_pos, void *dX, void *dW_gate, void *dW_up, void *dW_down,
                     void *dWs_gate, void *dWs_up, void *dWs_down, float *dlogits,
                     void *dW_router, void *ws, size_t ws_bytes, mok_stream_t stream);

/* The whole layer forward (route, dispatch, expert forward) with x and y in HOST memory:
 * copies x_host[T,d] (bf16) to the workspace, runs the layer and copies y back to
 * y_host[T,d].  Pinned host memory makes the copies asynchronous; the call returns without
 * waiting (synchronise the stream before reading y_host, or writing x_host again).  Routing
 * tensors live inside the workspace (mok_workspace_size(dims, MOK_PASS_FORWARD) +
 * mok_layer_host_extra_size(dims)).  The copy of x runs on a library-owned copy stream into one
 * of two device buffers of the workspace, alternating per call, so that a call's copy overlaps
 * the kernels of the previous call on the same workspace; `stream` waits for it before the
 * layer runs, so synchronising `stream` still covers the whole call.  The library keeps one
 * copy stream per device and two events per workspace (for the 16 most recent workspaces).
 * When y_host is pinned (mapped) host memory, the final combine writes y straight into it;
 * otherwise y is combined in the workspace and copied back on `stream`. */
size_t mok_layer_host_extra_size(const mok_dims *dims);
int mok_layer_forward_host(const mok_dims *dims, const mok_weights *w, const void *x_host,
                           void *y_host, void *ws, size_t ws_bytes, mok_stream_t stream);

/* Schedule of the bf16 expert GEMMs of mok_moe_forward (process-wide; default
 * MOK_SCHEDULE_TWO_LAUNCHES):
 *  - MOK_SCHEDULE_TWO_LAUNCHES: gate/up + SwiGLU, then down + router weight, each one persistent
 *    launch whose CTAs take the tiles c, c + grid, c + 2 grid, ...
 *  - MOK_SCHEDULE_FUSED: both phases in one persistent launch.  CTAs claim tiles in order from a
 *    device work counter (every gate/up tile before any down tile) and a down tile first waits,
 *    bounded, until every gate/up tile of its M tile has written its h rows (a readiness counter
 *    per M tile).  This is the fused, device-scheduled form of the layer's kernel (page
 *    "Mixture-of-Kittens: Nhân kernel MoE ...", intro and section "Lập lịch"; page
 *    "Mixture-of-Kittens; MoE megakernel", key points); on one GPU it measured about 1% slower
 *    than two launches at the DeepSeek-V3 shape, hence not the default.
 * Results are bit-identical under both.  Shapes run in CTA pairs (at least 320 routed rows per
 * expert) or with d % 256 != 0 always use two launches.  Returns MOK_OK, or MOK_ERR_INVALID_ARG
 * for another value; *previous (NULL to skip) receives the schedule before the call. */
typedef enum { MOK_SCHEDULE_TWO_LAUNCHES = 0, MOK_SCHEDULE_FUSED = 1 } mok_schedule;
int mok_set_forward_schedule(int schedule, int *previous);

/* Human-readable name of a status code (static string). */
const char *mok_status_string(int status);

/* Synchronises `stream`, copies the device status word of `ws` into *status_out (MOK_OK or a
 * negative code).  The one entry point that waits on the GPU. */
int mok_read_device_status(const void *ws, int *status_out, mok_stream_t stream);

/* Enqueues a reset of the device status word of `ws` to MOK_OK. */
int mok_clear_device_status(void *ws, mok_stream_t stream);

/* Number of kernel launches the last successful call of each entry point enqueued on this
 * host thread (for launch accounting in benchmarks). */
int mok_last_launch_count(void);

/* Pull schedule without a workspace: same inputs as mok_dispatch_index and, for valid inputs,
 * the same outputs, but the scratch it needs (a status word and the per-chunk expert histogram)
 * lives in a device array owned by the library (a 256-byte header plus a 1 MiB histogram), so
 * the call allocates nothing and takes no `ws`.  The pages describe no such variant; it exists
 * for callers that may not allocate device memory when they build the routing (a runtime that
 * reserves all memory at start-up, or code that must not trigger the device-wide
 * synchronisation of cudaMalloc/cudaFree).
 *  - Limit: E * ceil(T / 64) <= 262144 (T <= 65536 tokens at E = 256, T <= 32768 at E = 512);
 *    larger sizes return MOK_ERR_WORKSPACE and enqueue nothing.
 *  - The first call on each device looks up the array's device address (with that device
 *    current) and caches it; make that first call before any stream capture.
 *  - Every device holds the array until the process exits.  All calls on a device share it
 *    and it keeps the last call's contents, so calls whose GPU work overlaps (different
 *    streams, no ordering between them) race; order them on one stream.
 *  - Invalid routing is not reported: an expert index outside [0,E) drops that route
 *    (inv_pos = -1, offsets[E] < T*k), where mok_dispatch_index would also set
 *    MOK_ERR_DEVICE_CHECK in its workspace status word.  Callers that cannot vouch for their
 *    indices can compare offsets[E] with T*k. */
int mok_dispatch_index_noalloc(const mok_dims *dims, const int32_t *topk_idx, const float *topk_w,
                               int32_t *counts, int32_t *offsets, int32_t *sorted_tok,
                               float *sorted_w, int32_t *inv_pos, mok_stream_t stream);

/* Failure-detection self-test: launches one block that waits, with the library's bounded-wait
 * code and a budget of budget_ns (at most 2 s), on a barrier nothing arrives on.  The wait runs
 * out, MOK_ERR_TIMEOUT is recorded in the status word of `ws` and the kernel returns normally,
 * so the context stays usable.  It exercises the error path of the kernels' waits without
 * faulting or hanging the GPU. */
int mok_selftest_bounded_wait(void *ws, int64_t budget_ns, mok_stream_t stream);

/* Kernel timing for benchmarks.  While enabled on the calling host thread, every entry point
 * records a CUDA event pair around each kernel it launches, on the launch stream (the events do
 * not change what the GPU executes).  enable = 0 stops recording. */
int mok_timing_enable(int enable);

/* Waits for the recorded events, then returns per kernel name (up to max_kernels entries,
 * `names` holds max_kernels * 32 bytes, NUL-terminated) the number of launches and their summed
 * device time in milliseconds; *n_out = entries written.  Clears the record. */
int mok_timing_collect(char *names, int *launches, double *ms, int max_kernels, int *n_out);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H */
