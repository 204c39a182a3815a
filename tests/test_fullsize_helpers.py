"""The full-size test helpers on the CPU: exact bf16 bits -> float64, the expert-covering token
sample, and the oracle's per-expert work run in a spawn pool giving exactly the serial result."""

import numpy as np
import torch

import oracle
from mixture_experts_layer_14_gb300.synthetic import LayerShape, make_layer
from tests._fullsize import BF16Bits, cover_tokens, most_experts_tokens, oracle_pool
from tests._helpers import f64


def test_bf16_bits_convert_exactly():
    t = (torch.randn(64, 96) * torch.logspace(-20, 20, 96)).to(torch.bfloat16)
    b = BF16Bits(t.view(torch.int16).numpy().view(np.uint16))
    assert (np.asarray(b, dtype=np.float64) == t.to(torch.float64).numpy()).all()


def test_cover_tokens_reaches_every_selected_expert():
    rng = np.random.default_rng(0)
    idx = np.stack([rng.choice(64, size=4, replace=False) for _ in range(500)])
    idx[123] = [60, 61, 62, 63]                      # experts only token 123 selects
    idx[idx >= 60] = 59
    idx[123] = [60, 61, 62, 63]
    toks = cover_tokens(idx, 40, must=[0, 499])
    assert 123 in toks and 0 in toks and 499 in toks and len(toks) >= 40
    assert set(idx[toks].ravel().tolist()) == set(idx.ravel().tolist())
    m = most_experts_tokens(idx, 8)
    assert len(m) == 8 and len(set(idx[m].ravel().tolist())) >= 8 * 4 - 4


def test_pool_map_equals_serial_map():
    shape = LayerShape("pool_check", 48, 64, 6, 2, 64, 64, 1, 0.0, "zipf", "mxfp8", True, 62)
    L = make_layer(shape, "cpu", with_dy=True)
    x, dY, Wr, b = f64(L["x"]), f64(L["dY"]), f64(L["W_router"]), f64(L["bias"])
    l64 = oracle.router_logits(x, Wr, b)
    idx = oracle.topk_select(l64.astype(np.float32), shape.k)
    w = oracle.weights_for_selection(l64, idx)
    sh = (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))

    class Bits:
        def __init__(self, t):
            self.t = t

        def __getitem__(self, e):
            return BF16Bits(self.t[e].view(torch.int16).numpy().view(np.uint16))

    Wg, Wu, Wd = Bits(L["W_gate"]), Bits(L["W_up"]), Bits(L["W_down"])
    with oracle_pool(2) as pmap:
        y_mx = oracle.moe_forward_mxfp8(x, Wg, Wu, Wd, sh, idx, w, expert_map=pmap)
        y = oracle.moe_forward(x, Wg, Wu, Wd, sh, idx, w, expert_map=pmap)
        g = oracle.moe_backward_mxfp8(x, dY, Wr, Wg, Wu, Wd, sh, l64, idx, expert_map=pmap)
        g2 = oracle.moe_backward(x, dY, Wr, Wg, Wu, Wd, sh, l64, idx, weight_grads=False, expert_map=pmap)
    Wg64, Wu64, Wd64 = f64(L["W_gate"]), f64(L["W_up"]), f64(L["W_down"])
    assert (y_mx == oracle.moe_forward_mxfp8(x, Wg64, Wu64, Wd64, sh, idx, w)).all()
    assert (y == oracle.moe_forward(x, Wg64, Wu64, Wd64, sh, idx, w)).all()
    ref = oracle.moe_backward_mxfp8(x, dY, Wr, Wg64, Wu64, Wd64, sh, l64, idx)
    for key in ("dX", "dW_gate", "dW_up", "dW_down", "dlogits", "dw"):
        assert (g[key] == ref[key]).all(), key
    ref2 = oracle.moe_backward(x, dY, Wr, Wg64, Wu64, Wd64, sh, l64, idx)
    assert (g2["dX"] == ref2["dX"]).all() and g2["dW_gate"] is None
