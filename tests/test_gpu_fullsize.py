"""Parity at the full workload sizes, in the launch configuration bench.py times.

Routing, counts, offsets and the schedule are checked on every token against the oracle (cheap:
2 T d E flops).  The layer output is checked on at least 64 tokens chosen so that every active
expert is reached (the hottest one, and every expert that holds a single token, included),
whose rows the oracle computes one expert at a time in a process pool.  The backward is checked
on 32 tokens that reach as many experts as possible (dX, dlogits), on four experts in full (dW
over all their tokens: the hottest, the least busy non-empty one, a median one and one whose
rows end in a part-filled 128-row tile; dlogits of all those tokens and the four experts'
columns of dW_router), and on the shared expert's weight gradients."""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, make_layer
from tests._fullsize import dw_experts, experts_of, most_experts_tokens, oracle_pool, sampled_tokens
from tests._helpers import NEAR_TIE, assert_close, dims_of, ensure_lib, f64

pytestmark = pytest.mark.gpu


def route_checks(shape, L, layer):
    """Selection (bit-exact off near ties), counts, offsets, schedule and weights on all tokens."""
    x64 = f64(L["x"])
    Wr = f64(L["W_router"])
    b = None if L["bias"] is None else f64(L["bias"])
    l64 = oracle.router_logits(x64, Wr, b)
    l32 = l64.astype(np.float32)
    idx_ref = oracle.topk_select(l32, shape.k)
    got = layer.routing["topk_idx"].cpu().numpy()
    ok = oracle.topk_gap(l32, shape.k) >= NEAR_TIE
    assert (np.sort(got[ok], 1) == np.sort(idx_ref[ok], 1)).all()
    n_near = int((~ok).sum())
    counts, offsets, sorted_tok, inv_pos = oracle.dispatch(got, shape.E)
    assert (layer.routing["counts"].cpu().numpy() == counts).all()
    assert (layer.routing["offsets"].cpu().numpy() == offsets).all()
    assert (layer.routing["sorted_tok"].cpu().numpy() == sorted_tok).all()
    assert (layer.routing["inv_pos"].cpu().numpy() == inv_pos).all()
    w_ref = oracle.weights_for_selection(l64, got)
    np.testing.assert_allclose(layer.routing["topk_w"].cpu().numpy(), w_ref, rtol=1e-4, atol=1e-6)
    return x64, Wr, l64, got, counts, n_near


def shared_of(L):
    return (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))


@pytest.mark.parametrize("name", ["dsv3_bf16_fwd", "kimi_skew_bf16_fwd", "dsv3_decode_t64"])
def test_fullsize_forward(name):
    ensure_lib()
    shape = WORKLOADS[name]
    L = make_layer(shape, "cuda")
    layer = mok.MoELayer(dims_of(shape), L)
    y = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0
    x64, Wr, l64, got, counts, n_near = route_checks(shape, L, layer)
    toks = sampled_tokens(got, counts, shape.T)
    print(f"{name}: near-tie tokens excluded {n_near}; hottest expert {counts.max()} rows "
          f"(mean {counts.mean():.1f}); empty experts {(counts == 0).sum()}; {len(toks)} sampled "
          f"tokens reach all {(counts > 0).sum()} active experts")
    w_ref = oracle.weights_for_selection(l64[toks], got[toks])
    Wg, Wu, Wd = experts_of(L)
    with oracle_pool() as pmap:
        y_ref = oracle.moe_forward(x64[toks], Wg, Wu, Wd, shared_of(L), got[toks], w_ref, expert_map=pmap)
    mx, mn = assert_close("y sampled", f64(y[toks]), y_ref)
    print(f"{name}: y on {len(toks)} tokens max_rel {mx:.2e} mean_rel {mn:.2e}")
    # bit-identical rerun, and the same output from the fused schedule (where it applies)
    y2 = layer.forward(L["x"])
    prev = mok.set_forward_schedule(mok.SCHEDULE_FUSED)
    try:
        y3 = layer.forward(L["x"])
        torch.cuda.synchronize()
    finally:
        mok.set_forward_schedule(prev)
    assert mok.read_status(layer.ws) == 0
    assert torch.equal(y, y2) and torch.equal(y, y3)


def test_fullsize_training_backward():
    ensure_lib()
    shape = WORKLOADS["dsv3_bf16_train"]
    L = make_layer(shape, "cuda", with_dy=True)
    layer = mok.MoELayer(dims_of(shape), L)
    layer.forward(L["x"], training=True)
    g = layer.backward(L["x"], L["dY"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0 and mok.read_status(layer._ws_bwd) == 0
    x64, Wr, l64, got, counts, _ = route_checks(shape, L, layer)
    dY = L["dY"]
    Wg, Wu, Wd = experts_of(L)
    sh = shared_of(L)
    toks = most_experts_tokens(got, 32)
    picks = dw_experts(counts)
    with oracle_pool() as pmap:
        # dX and dlogits on sampled tokens (per-token quantities)
        ref = oracle.moe_backward(x64[toks], f64(dY[toks]), Wr, Wg, Wu, Wd, sh, l64[toks], got[toks],
                                  weight_grads=False, expert_map=pmap)
        # dW of four experts in full: all tokens routed to them, one pool job per expert
        rows = np.nonzero(np.isin(got, picks).any(1))[0]
        rw = oracle.moe_backward(x64[rows], f64(dY[rows]), Wr, Wg, Wu, Wd, None, l64[rows], got[rows],
                                 only_experts=picks, expert_map=pmap)
        # every expert of those tokens: their dlogits, and the columns of dW_router = x^T dl of
        # the four experts (all tokens with a nonzero dl in such a column are in these rows)
        rr = oracle.moe_backward(x64[rows], f64(dY[rows]), Wr, Wg, Wu, Wd, sh, l64[rows], got[rows],
                                 weight_grads=False, expert_map=pmap)
    n_exp = len(set(got[toks].ravel().tolist()))
    assert_close("dX sampled", f64(g["dX"][toks]), ref["dX"])
    assert_close("dlogits sampled", f64(g["dlogits"][toks]), ref["dlogits"])
    print(f"dX, dlogits on {len(toks)} tokens reaching {n_exp} experts; dW in full for experts "
          f"{picks} with {[int(counts[e]) for e in picks]} rows")
    for e in picks:
        for key in ("dW_gate", "dW_up", "dW_down"):
            assert_close(f"{key}[{e}]", f64(g[key][e]), rw[key][e])
    # shared expert weight gradients over all tokens (the oracle with no routed-expert terms)
    rs = oracle.moe_backward(x64, f64(dY), Wr, Wg, Wu, Wd, sh, l64, got, only_experts=[])
    for key in ("dWs_gate", "dWs_up", "dWs_down"):
        assert_close(key, f64(g[key]), rs[key])
    assert_close("dlogits of those tokens", f64(g["dlogits"][rows]), rr["dlogits"])
    assert_close("dW_router columns", f64(g["dW_router"][:, picks]), rr["dW_router"][:, picks])
    # dW_router = x^T dlogits over all tokens: consistent with the GPU's own dlogits
    assert_close("dW_router vs x^T dlogits", f64(g["dW_router"]), x64.T @ f64(g["dlogits"]))
    assert_dlogit_rows_sum_to_zero(g["dlogits"])


def assert_dlogit_rows_sum_to_zero(dlogits):
    """Every token's logit gradient sums to zero: dl_m = w_m (dw_m - sum_j w_j dw_j) over the
    selection and sum_m w_m = 1 (the renormalised softmax), a property of all T tokens."""
    dl = f64(dlogits)
    scale = np.abs(dl).sum(axis=1)
    assert (np.abs(dl.sum(axis=1)) <= 1e-4 * scale + 1e-30).all()
