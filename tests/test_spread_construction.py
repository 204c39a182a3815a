"""The magnitude-spread construction of the MXFP8 GPU parity cases (tests/_spread.py), on the
CPU: the float64 oracle's outputs and gradients of the spread layer, unscaled, equal those of
the original layer, so the spread changes only where the MXFP8 reading rounds."""

import numpy as np

import oracle
from mixture_experts_layer_14_gb300.synthetic import LayerShape, make_layer
from tests._helpers import f64
from tests._spread import apply_spread, spread_factors, unscale


def test_spread_layer_is_the_same_float64_function():
    shape = LayerShape("spread_check", 40, 64, 4, 2, 64, 32, 1, 0.0, "zipf", "mxfp8", True, 61)
    L = make_layer(shape, "cpu", with_dy=True)
    s = spread_factors(shape, 9, 1)
    S = apply_spread(L, s)

    def run(M):
        x, Wr, b = f64(M["x"]), f64(M["W_router"]), f64(M["bias"])
        logits = oracle.router_logits(x, Wr, b)
        idx = oracle.topk_select(logits.astype(np.float32), shape.k)
        w = oracle.weights_for_selection(logits, idx)
        sh = (f64(M["Ws_gate"]), f64(M["Ws_up"]), f64(M["Ws_down"]))
        Wg, Wu, Wd = f64(M["W_gate"]), f64(M["W_up"]), f64(M["W_down"])
        y = oracle.moe_forward(x, Wg, Wu, Wd, sh, idx, w)
        g = oracle.moe_backward(x, f64(M["dY"]), Wr, Wg, Wu, Wd, sh, logits, idx)
        return idx, y, g

    idx0, y0, g0 = run(L)
    idx1, y1, g1 = run(S)
    assert (idx0 == idx1).all()
    # the spread tensors really mix magnitudes 2^18 apart along each axis
    assert np.ptp(s["r"]) == 18 and np.ptp(s["c"]) == 18
    assert np.allclose(unscale("y", y1, s), y0, rtol=1e-9, atol=1e-12 * np.abs(y0).max())
    for key in ("dX", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down", "dlogits",
                "dW_router"):
        ref = g0[key]
        assert np.allclose(unscale(key, g1[key], s), ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max()), key
