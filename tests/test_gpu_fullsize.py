"""Parity at the full workload sizes, in the launch configuration bench.py times.

Routing, counts, offsets and the schedule are checked on every token against the oracle (cheap:
2 T d E flops).  The layer output is checked on sampled tokens, whose rows the oracle computes
one by one.  The backward is checked on sampled tokens (dX, dlogits) and on sampled experts in
full (dW over all their tokens), plus the shared expert's weight gradients."""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, make_layer
from tests._helpers import NEAR_TIE, LazyExperts, assert_close, dims_of, ensure_lib, f64

pytestmark = pytest.mark.gpu


def _route_checks(shape, L, layer):
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


def _shared(L):
    return (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))


@pytest.mark.parametrize("name,samples", [("dsv3_bf16_fwd", 4), ("kimi_skew_bf16_fwd", 4),
                                          ("dsv3_decode_t64", 4)])
def test_fullsize_forward(name, samples):
    ensure_lib()
    shape = WORKLOADS[name]
    L = make_layer(shape, "cuda")
    layer = mok.MoELayer(dims_of(shape), L)
    y = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0
    x64, Wr, l64, got, counts, n_near = _route_checks(shape, L, layer)
    print(f"{name}: near-tie tokens excluded {n_near}; hottest expert {counts.max()} rows "
          f"(mean {counts.mean():.1f}); empty experts {(counts == 0).sum()}")
    # sampled tokens: include one routed to the hottest expert
    hot = int(np.argmax(counts))
    toks = [0, shape.T - 1, int(np.nonzero((got == hot).any(1))[0][0]), shape.T // 2][:samples]
    w_ref = oracle.weights_for_selection(l64[toks], got[toks])
    y_ref = oracle.moe_forward(x64[toks], LazyExperts(L["W_gate"]), LazyExperts(L["W_up"]),
                               LazyExperts(L["W_down"]), _shared(L), got[toks], w_ref)
    assert_close("y sampled", f64(y[toks]), y_ref)
    # bit-identical rerun
    y2 = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_fullsize_training_backward():
    ensure_lib()
    shape = WORKLOADS["dsv3_bf16_train"]
    L = make_layer(shape, "cuda", with_dy=True)
    layer = mok.MoELayer(dims_of(shape), L)
    layer.forward(L["x"], training=True)
    g = layer.backward(L["x"], L["dY"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0 and mok.read_status(layer._ws_bwd) == 0
    x64, Wr, l64, got, counts, _ = _route_checks(shape, L, layer)
    dY = L["dY"]
    Wg, Wu, Wd = LazyExperts(L["W_gate"]), LazyExperts(L["W_up"]), LazyExperts(L["W_down"])
    sh = _shared(L)
    # dX and dlogits on sampled tokens (per-token quantities)
    toks = [0, 1, shape.T - 1]
    ref = oracle.moe_backward(x64[toks], f64(dY[toks]), Wr, Wg, Wu, Wd, sh, l64[toks], got[toks])
    assert_close("dX sampled", f64(g["dX"][toks]), ref["dX"])
    assert_close("dlogits sampled", f64(g["dlogits"][toks]), ref["dlogits"])
    # dW of two experts in full: all tokens routed to them
    for e in (int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))):
        rows = np.nonzero((got == e).any(1))[0]
        r = oracle.moe_backward(x64[rows], f64(dY[rows]), Wr, Wg, Wu, Wd, None, l64[rows], got[rows],
                                only_experts=[e])
        assert_close(f"dW_gate[{e}]", f64(g["dW_gate"][e]), r["dW_gate"][e])
        assert_close(f"dW_up[{e}]", f64(g["dW_up"][e]), r["dW_up"][e])
        assert_close(f"dW_down[{e}]", f64(g["dW_down"][e]), r["dW_down"][e])
    # shared expert weight gradients over all tokens (the oracle with no routed-expert terms)
    rs = oracle.moe_backward(x64, f64(dY), Wr, Wg, Wu, Wd, sh, l64, got, only_experts=[])
    for key in ("dWs_gate", "dWs_up", "dWs_down"):
        assert_close(key, f64(g[key]), rs[key])
    # dW_router = x^T dlogits: consistent with the GPU's own dlogits (property at full size)
    assert_close("dW_router vs x^T dlogits", f64(g["dW_router"]), x64.T @ f64(g["dlogits"]))
    _assert_dlogit_rows_sum_to_zero(g["dlogits"])


def _assert_dlogit_rows_sum_to_zero(dlogits):
    """Every token's logit gradient sums to zero: dl_m = w_m (dw_m - sum_j w_j dw_j) over the
    selection and sum_m w_m = 1 (the renormalised softmax), a property of all T tokens."""
    dl = f64(dlogits)
    scale = np.abs(dl).sum(axis=1)
    assert (np.abs(dl.sum(axis=1)) <= 1e-4 * scale + 1e-30).all()
