"""Float64 reference of the MoE layer: router, top-k, pull schedule, SwiGLU experts, combine,
and the backward pass.  Test infrastructure only (see the package docstring).

Layouts follow the problem statement of the layer: x[T,d], W_router[d,E], per routed expert
W_gate/W_up[d,F] and W_down[F,d] (stacked as [E,d,F] / [E,F,d]), shared expert
Ws_gate/Ws_up[d,Fs], Ws_down[Fs,d].  Row vectors: g = x @ W_gate.

Every floating-point quantity is computed in float64 from the (bf16-exact) inputs and is not
rounded to a narrower type, except the router logits used for the *top-k decision*, which are
rounded to float32 first because the GPU takes that integer decision on float32 logits.
"""

import numpy as np


def to_f64(a):
    """Exact conversion of a bf16/fp32/fp64 array (numpy or CPU torch tensor) to float64."""
    try:
        import torch  # only for accepting CPU tensors; no arithmetic of the method

        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Router.  Page "Mixture-of-Kittens: Nhân kernel MoE ...", section "Chồng lấp tính toán và
# truyền tải trong MoE": a router projection selects the top-k routed experts per token and
# assigns each a router weight.  Plain reading: logits = x @ W_router + b, softmax over all
# experts, top-k on the logits (descending, ties to the lower expert index), weights are the
# selected probabilities renormalised to sum to one.
# --------------------------------------------------------------------------------------

def router_logits(x, W_router, bias=None):
    """l[t,e] = sum_i x[t,i] W_router[i,e] + b[e], float64.  Pinned via the top-k and weight
    pins (brute-force subsets, softmax identities) and the finite-difference pin of dW_router."""
    l = x @ W_router
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def topk_select(logits32, k):
    """Indices of the k largest float32 logits per row, in order (logit descending, expert
    index ascending among equal logits).  Pinned against brute-force enumeration of all
    k-subsets in tests."""
    l32 = np.asarray(logits32, dtype=np.float32)
    # stable sort of the negated values keeps equal logits in ascending index order
    order = np.argsort(-l32, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def topk_gap(logits32, k):
    """Gap between the k-th and (k+1)-th largest float32 logit of each row (inf when k == E).
    Tokens with a gap below 1e-4 are near ties whose selection is not compared bit-exactly."""
    l32 = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    E = l32.shape[1]
    if k >= E:
        return np.full(l32.shape[0], np.inf)
    s = -np.sort(-l32, axis=1)
    return s[:, k - 1] - s[:, k]


def weights_for_selection(logits, topk_idx):
    """w_j = p[e_j] / sum_{i in selection} p[e_i] with p = softmax(logits) over all experts.
    Pinned by the closed-form identity w = softmax over the selected logits only, sum w = 1,
    and k = E giving w = p."""
    l = np.asarray(logits, dtype=np.float64)
    m = l.max(axis=1, keepdims=True)
    ex = np.exp(l - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, np.asarray(topk_idx, dtype=np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(x, W_router, bias, k):
    """Router of the layer.  Returns (logits64, logits32, topk_idx, topk_w)."""
    l64 = router_logits(x, W_router, bias)
    l32 = l64.astype(np.float32)
    idx = topk_select(l32, k)
    w = weights_for_selection(l64, idx)
    return l64, l32, idx, w


# --------------------------------------------------------------------------------------
# Pull schedule.  Page "Mixture-of-Kittens: Nhân kernel MoE ...", section "Lập lịch": the
# schedule is built without a sort by scanning the routing tensor and appending every route
# that targets a (local) expert; outputs are tokens per expert, region offsets and a table
# whose row is the destination row.  On one GPU every expert is local and the source rank is 0.
# Page "Метод и эксперименты": each expert then reads its own tokens, e.g. E2 <- [0,2,9,15].
# --------------------------------------------------------------------------------------

def dispatch(topk_idx, E):
    """Returns counts[E], offsets[E+1] (exclusive prefix sum), sorted_tok[T*k] (token of each
    destination row; tokens ascending inside an expert's region) and inv_pos[T,k] (destination
    row of route (t,j)).  Pinned by the worked example fixture and permutation checks."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    sorted_tok = np.zeros(T * k, dtype=np.int64)
    inv_pos = np.zeros((T, k), dtype=np.int64)
    for t in range(T):  # scanning tokens in order appends them in ascending order per expert
        for j in range(k):
            e = idx[t, j]
            pos = fill[e]
            fill[e] += 1
            sorted_tok[pos] = t
            inv_pos[t, j] = pos
    return (counts.astype(np.int32), offsets.astype(np.int32),
            sorted_tok.astype(np.int32), inv_pos.astype(np.int32))


# --------------------------------------------------------------------------------------
# Expert FFN.  Same page, section "Chồng lấp tính toán ...": up and gate projections, SwiGLU
# activation, down projection.  SiLU(z) = z * sigmoid(z).
# --------------------------------------------------------------------------------------

def silu(z):
    """z / (1 + exp(-z)).  Pinned at closed-form points (0, +-ln 3, large |z|)."""
    return z / (1.0 + np.exp(-z))


def expert_ffn(X, Wg, Wu, Wd):
    """SwiGLU FFN of one expert on rows X[n,d]: g = X Wg, u = X Wu, h = SiLU(g) u, y = h Wd.
    Returns (g, u, h, y).  Pinned with permutation-matrix weights (closed form) and
    linearity/zero-gate invariants."""
    g = X @ Wg
    u = X @ Wu
    h = silu(g) * u
    return g, u, h, h @ Wd


# --------------------------------------------------------------------------------------
# Layer forward.  y[t] = shared(x_t) + sum_j w_j y_{e_j}(x_t).
# --------------------------------------------------------------------------------------

def _experts_used(topk_idx):
    return sorted(set(int(e) for e in np.asarray(topk_idx).ravel()))


def _ffn_rows(job):
    """Output rows of one expert's FFN (a module-level function so that a process pool can
    run it)."""
    X, Wg_e, Wu_e, Wd_e = job
    return expert_ffn(X, np.asarray(Wg_e, dtype=np.float64), np.asarray(Wu_e, dtype=np.float64),
                      np.asarray(Wd_e, dtype=np.float64))[3]


def moe_forward(x, Wg, Wu, Wd, shared, topk_idx, topk_w, expert_map=map):
    """Layer output for the rows of x.  ``Wg/Wu/Wd`` are indexable by expert id (a stacked
    array or any lazy accessor returning [d,F] / [F,d] matrices convertible to float64);
    ``shared`` is (Ws_gate, Ws_up, Ws_down) or None; ``expert_map`` runs the per-expert work
    (``map`` or a pool's ``imap``).  Pinned by: k = E with identical experts reduces to
    shared + FFN; token permutation permutes outputs; a zero router weight contributes nothing;
    E = k = 1 gives shared + FFN."""
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    y = np.zeros_like(x)
    if shared is not None:
        y += expert_ffn(x, *shared)[3]
    experts = _experts_used(idx)
    sel = [np.nonzero(idx == e) for e in experts]
    jobs = ((x[rows], Wg[e], Wu[e], Wd[e]) for e, (rows, _) in zip(experts, sel))
    for (rows, slots), ye in zip(sel, expert_map(_ffn_rows, jobs)):  # float64: order is moot
        np.add.at(y, rows, w[rows, slots][:, None] * ye)
    return y


def moe_forward_from_logits(x, logits, topk_idx, Wg, Wu, Wd, shared):
    """Forward with the selection held fixed and the weights recomputed from ``logits``
    (used for finite differences with respect to the logits and the router weights)."""
    w = weights_for_selection(logits, topk_idx)
    return moe_forward(x, Wg, Wu, Wd, shared, topk_idx, w)


# --------------------------------------------------------------------------------------
# Backward.  Gradients of L = sum(dY * y) with the top-k selection held constant; experts that
# a token did not select get no gradient from it.  Pinned by central finite differences.
# --------------------------------------------------------------------------------------

def _ffn_backward(job):
    """Backward of one SwiGLU FFN on rows X with upstream dYr and router weights wr (a
    module-level function so that a process pool can run it).  Returns (dX rows, dW_gate,
    dW_up, dW_down, dw rows); the weight gradients are None unless job[-1] (weight_grads)."""
    X, dYr, wr, Wge, Wue, Wde, weight_grads = job
    Wge = np.asarray(Wge, dtype=np.float64)
    Wue = np.asarray(Wue, dtype=np.float64)
    Wde = np.asarray(Wde, dtype=np.float64)
    g = X @ Wge
    u = X @ Wue
    s = 1.0 / (1.0 + np.exp(-g))
    h = g * s * u
    a = dYr @ Wde.T                      # dL/d(h) before the router weight
    dwr = (a * h).sum(axis=1)            # <dY, h Wd> = <a, h>
    dh = wr[:, None] * a
    dg = dh * u * s * (1.0 + g * (1.0 - s))   # d SiLU(g)/dg = s (1 + g (1 - s))
    du = dh * g * s
    dXr = dg @ Wge.T + du @ Wue.T
    if not weight_grads:
        return dXr, None, None, None, dwr
    return dXr, X.T @ dg, X.T @ du, (wr[:, None] * h).T @ dYr, dwr


def moe_backward(x, dY, W_router, Wg, Wu, Wd, shared, logits, topk_idx, only_experts=None,
                 weight_grads=True, expert_map=map):
    """``only_experts`` (optional) restricts the routed-expert terms to those expert ids (for
    checks of sampled experts on large inputs; dX and the router terms are then partial).
    ``weight_grads=False`` skips the weight gradients (returned as None); ``expert_map`` runs the
    per-expert work (``map``, or a process pool's ``imap`` for large layers).
    Returns a dict with dX[T,d], dW_gate/dW_up[E,d,F], dW_down[E,F,d], dWs_gate/dWs_up[d,Fs],
    dWs_down[Fs,d] (None without a shared expert), dlogits[T,E], dW_router[d,E] and the
    per-route router-weight gradients dw[T,k] (= <dY_t, y_{e_j}(x_t)>)."""
    x = np.asarray(x, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    Wr = np.asarray(W_router, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, d = x.shape
    E = Wr.shape[1]
    k = idx.shape[1]
    w = weights_for_selection(logits, idx)
    dX = np.zeros_like(x)
    # per-expert gradients; stacked into [E, ...] arrays unless only some experts are asked for
    dWg, dWu, dWd = {}, {}, {}
    dw = np.zeros((T, k))

    sel = [(e,) + np.nonzero(idx == e) for e in (range(E) if only_experts is None else only_experts)]
    sel = [t for t in sel if t[1].size]
    jobs = ((x[rows], dY[rows], w[rows, slots], Wg[e], Wu[e], Wd[e], weight_grads)
            for e, rows, slots in sel)
    for (e, rows, slots), (dXr, dWg[e], dWu[e], dWd[e], dwr) in zip(sel, expert_map(_ffn_backward, jobs)):
        np.add.at(dX, rows, dXr)
        dw[rows, slots] = dwr

    dWs = None
    if shared is not None:
        dXs, dWsg, dWsu, dWsd, _ = _ffn_backward((x, dY, np.ones(T), *shared, weight_grads))
        dX += dXs
        dWs = (dWsg, dWsu, dWsd)

    # w_j = exp(l_j) / sum_{i in S} exp(l_i)  =>  dl_m = w_m (dw_m - sum_j w_j dw_j), m in S
    dl = np.zeros((T, E))
    inner = (w * dw).sum(axis=1, keepdims=True)
    np.put_along_axis(dl, idx, w * (dw - inner), axis=1)
    dX += dl @ Wr.T
    dWr = x.T @ dl
    if not weight_grads:
        dWg = dWu = dWd = None
    elif only_experts is None:
        Wg0 = np.asarray(Wg[0], dtype=np.float64)
        zg = np.zeros(Wg0.shape)
        zd = np.zeros(Wg0.shape[::-1])
        dWg = np.stack([dWg.get(e, zg) for e in range(E)])
        dWu = np.stack([dWu.get(e, zg) for e in range(E)])
        dWd = np.stack([dWd.get(e, zd) for e in range(E)])
    return {
        "dX": dX, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd,
        "dWs_gate": None if dWs is None else dWs[0],
        "dWs_up": None if dWs is None else dWs[1],
        "dWs_down": None if dWs is None else dWs[2],
        "dlogits": dl, "dW_router": dWr, "dw": dw,
    }


# --------------------------------------------------------------------------------------
# MXFP8 reading of the forward (page "Mixture-of-Kittens; MoE megakernel", key points: the kernel
# supports BF16 and MXFP8).  x, every expert weight (blocks of 32 along its reduction
# dimension) and h (along F) pass through E4M3/UE8M0 quantise-dequantise; the router, the
# weighting and the combine stay in full precision; products and sums are float64.
# --------------------------------------------------------------------------------------

def _mx_qd(a):
    from .mxfp8 import mx_dequantize, mx_quantize

    q, sc = mx_quantize(a)
    return mx_dequantize(q, sc)


def _mx_weight(W):
    """[K, N] weight quantised along K (its reduction dimension), returned as [K, N]."""
    return _mx_qd(np.asarray(W, dtype=np.float64).T).T


def _mx_ffn(job):
    """One expert's FFN at the MXFP8 quantisation points, on rows X that are already quantised
    (a module-level function so that a process pool can run it): g and u from weights quantised
    along d, h quantised along F, then the down projection with its weight quantised along F."""
    X, Wg_e, Wu_e, Wd_e = job
    g = X @ _mx_weight(Wg_e)
    u = X @ _mx_weight(Wu_e)
    h = _mx_qd(silu(g) * u)
    return h @ _mx_weight(Wd_e)


def moe_forward_mxfp8(x, Wg, Wu, Wd, shared, topk_idx, topk_w, expert_map=map):
    """Layer output with the MXFP8 quantisation points of the path.  A composition of the
    pinned quantiser and FFN pieces; pinned further by: values exactly representable in MXFP8
    are fixed points of the quantiser, zero down weights give a zero output, the distance to
    moe_forward on random data stays within a few E4M3 steps, and the locality pins of every
    quantisation axis.  ``expert_map`` runs the per-expert work (``map`` or a pool's ``imap``)."""
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    xq = _mx_qd(x)

    y = np.zeros_like(x)
    if shared is not None:
        y += _mx_ffn((xq, *shared))
    experts = _experts_used(idx)
    sel = [np.nonzero(idx == e) for e in experts]
    jobs = ((xq[rows], Wg[e], Wu[e], Wd[e]) for e, (rows, _) in zip(experts, sel))
    for (rows, slots), ye in zip(sel, expert_map(_mx_ffn, jobs)):
        np.add.at(y, rows, w[rows, slots][:, None] * ye)
    return y


# --------------------------------------------------------------------------------------
# MXFP8 reading of the backward.  The pages give MXFP8 for the layer's kernel without saying
# which GEMMs of a training step it covers; the plain extension of the forward reading above is
# taken: every expert GEMM of the backward multiplies E4M3/UE8M0 operands, each quantised in
# blocks of 32 along that GEMM's own reduction dimension, with exact products and sums:
#   a       = q_d(dY) q_d(W_down)^T                       (reduction over d)
#   dX_e    = q_F(dG) q_F(W_gate)^T + q_F(dU) q_F(W_up)^T    (over F)
#   dW_gate = q_t(X)^T q_t(dG),  dW_up = q_t(X)^T q_t(dU),  dW_down = q_t(w h)^T q_t(dY)
#             (over the expert's tokens, in token order, blocks of 32 from its first token)
# The forward values being differentiated are those of the MXFP8 forward (g = q_d(x) q_d(W_gate),
# u likewise).  The router terms (dl W_router^T, x^T dl), the SwiGLU derivative and the
# router-weight gradient <a, h> stay unquantised.
# --------------------------------------------------------------------------------------

def _mx_qd_tokens(A):
    """Quantise-dequantise A[n, C] along its first axis (tokens) in blocks of 32 rows from row 0;
    a last partial block counts as padded with zeros (zeros do not change a block's amax)."""
    A = np.asarray(A, dtype=np.float64)
    n = A.shape[0]
    pad = (-n) % 32
    Ap = np.concatenate([A, np.zeros((pad,) + A.shape[1:])], axis=0)
    return _mx_qd(Ap.T).T[:n]


def _mx_ffn_backward(job):
    """Backward of one expert's FFN at the MXFP8 quantisation points (a module-level function so
    that a process pool can run it).  X, Xq: its rows of x and of q_d(x); dYr, dYrq likewise for
    dY; wr its router weights.  Returns (dX rows, dW_gate, dW_up, dW_down, dw rows); the weight
    gradients are None unless job[-1] (weight_grads)."""
    X, Xq, dYr, dYrq, wr, Wge, Wue, Wde, weight_grads = job
    Wge = np.asarray(Wge, dtype=np.float64)
    Wue = np.asarray(Wue, dtype=np.float64)
    Wde = np.asarray(Wde, dtype=np.float64)
    g = Xq @ _mx_weight(Wge)                 # the MXFP8 forward's gate and up values
    u = Xq @ _mx_weight(Wue)
    s = 1.0 / (1.0 + np.exp(-g))
    h = g * s * u
    a = dYrq @ _mx_qd(Wde).T                 # W_down [F, d]: blocks along d
    dwr = (a * h).sum(axis=1)
    dh = wr[:, None] * a
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    dXr = _mx_qd(dg) @ _mx_qd(Wge).T + _mx_qd(du) @ _mx_qd(Wue).T   # W_gate [d, F]: along F
    if not weight_grads:
        return dXr, None, None, None, dwr
    hw = wr[:, None] * h
    Xt = _mx_qd_tokens(X)
    dWge = Xt.T @ _mx_qd_tokens(dg)
    dWue = Xt.T @ _mx_qd_tokens(du)
    dWde = _mx_qd_tokens(hw).T @ _mx_qd_tokens(dYr)
    return dXr, dWge, dWue, dWde, dwr


def moe_backward_mxfp8(x, dY, W_router, Wg, Wu, Wd, shared, logits, topk_idx, only_experts=None,
                       weight_grads=True, expert_map=map):
    """Gradients with the MXFP8 quantisation points above; same arguments and result keys as
    moe_backward.  Pinned by: every gradient stays within a few E4M3 steps of moe_backward's
    (itself pinned by finite differences) and differs from it; on inputs and weights exactly
    representable in MXFP8 the router-weight gradients, dlogits and dW_router equal the float64
    ones; the token-axis quantiser matches the pinned quantiser applied column by column; and
    by locality pins of every quantisation axis (an outlier coarsens only the values of its own
    block along that GEMM's reduction dimension)."""
    x = np.asarray(x, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    Wr = np.asarray(W_router, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, d = x.shape
    E = Wr.shape[1]
    k = idx.shape[1]
    w = weights_for_selection(logits, idx)
    xq = _mx_qd(x)
    dYq = _mx_qd(dY)
    dX = np.zeros_like(x)
    dWg, dWu, dWd = {}, {}, {}
    dw = np.zeros((T, k))

    sel = [(e,) + np.nonzero(idx == e) for e in (range(E) if only_experts is None else only_experts)]
    sel = [t for t in sel if t[1].size]
    jobs = ((x[rows], xq[rows], dY[rows], dYq[rows], w[rows, slots], Wg[e], Wu[e], Wd[e], weight_grads)
            for e, rows, slots in sel)
    for (e, rows, slots), (dXr, dWg[e], dWu[e], dWd[e], dwr) in zip(sel, expert_map(_mx_ffn_backward, jobs)):
        np.add.at(dX, rows, dXr)
        dw[rows, slots] = dwr

    dWs = None
    if shared is not None:
        dXs, dWsg, dWsu, dWsd, _ = _mx_ffn_backward((x, xq, dY, dYq, np.ones(T), *shared, weight_grads))
        dX += dXs
        dWs = (dWsg, dWsu, dWsd)

    dl = np.zeros((T, E))
    inner = (w * dw).sum(axis=1, keepdims=True)
    np.put_along_axis(dl, idx, w * (dw - inner), axis=1)
    dX += dl @ Wr.T
    dWr = x.T @ dl
    if not weight_grads:
        dWg = dWu = dWd = None
    elif only_experts is None:
        Wg0 = np.asarray(Wg[0], dtype=np.float64)
        zg = np.zeros(Wg0.shape)
        zd = np.zeros(Wg0.shape[::-1])
        dWg = np.stack([dWg.get(e, zg) for e in range(E)])
        dWu = np.stack([dWu.get(e, zg) for e in range(E)])
        dWd = np.stack([dWd.get(e, zd) for e in range(E)])
    return {
        "dX": dX, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd,
        "dWs_gate": None if dWs is None else dWs[0],
        "dWs_up": None if dWs is None else dWs[1],
        "dWs_down": None if dWs is None else dWs[2],
        "dlogits": dl, "dW_router": dWr, "dw": dw,
    }


# --------------------------------------------------------------------------------------
# NVFP4 reading of the forward (a NEXT variant: the pages name NVFP4 only as the format of
# their authors' earlier kernels).  Each expert GEMM multiplies NVFP4 operands quantised along
# its own reduction dimension, with the format and recipe of oracle/nvfp4.py: x and every
# gate/up weight along d, h and every down weight along F.  Weights carry their own tensor
# scale (per expert and projection, from the weight's amax); the activations x and h take a
# calibrated tensor amax given with the layer (amax_x, amax_h), the static form of the
# per-tensor scale, so a value above it saturates.  h is quantised from its fp32 value.  The
# router, the weighting and the combine stay in full precision; products and sums are float64.
# --------------------------------------------------------------------------------------

def _nv_qd(a, tensor_amax=None):
    from .nvfp4 import nv_dequantize, nv_quantize

    q, sc, g = nv_quantize(a, tensor_amax)
    return nv_dequantize(q, sc, g)


def _nv_weight(W):
    """[K, N] weight quantised along K (its reduction dimension) with its own tensor scale,
    returned as [K, N]."""
    return _nv_qd(np.asarray(W, dtype=np.float64).T).T


def _nv_ffn(job):
    """One expert's FFN at the NVFP4 quantisation points, on rows X that are already quantised
    (a module-level function so that a process pool can run it)."""
    X, Wg_e, Wu_e, Wd_e, amax_h = job
    g = X @ _nv_weight(Wg_e)
    u = X @ _nv_weight(Wu_e)
    h = _nv_qd(silu(g) * u, amax_h)
    return h @ _nv_weight(Wd_e)


def moe_forward_nvfp4(x, Wg, Wu, Wd, shared, topk_idx, topk_w, amax_x, amax_h, expert_map=map):
    """Layer output with the NVFP4 quantisation points of the path; ``amax_x`` and ``amax_h``
    are the calibrated tensor amaxes of the two activations.  A composition of the pinned
    quantiser and FFN pieces; pinned further by the axis pins of tests/test_oracle_nvfp4.py
    (which values an outlier coarsens), zero down weights, and the distance to moe_forward on
    random data."""
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    xq = _nv_qd(x, amax_x)

    y = np.zeros_like(x)
    if shared is not None:
        y += _nv_ffn((xq, *shared, amax_h))
    experts = _experts_used(idx)
    sel = [np.nonzero(idx == e) for e in experts]
    jobs = ((xq[rows], Wg[e], Wu[e], Wd[e], amax_h) for e, (rows, _) in zip(experts, sel))
    for (rows, slots), ye in zip(sel, expert_map(_nv_ffn, jobs)):
        np.add.at(y, rows, w[rows, slots][:, None] * ye)
    return y
