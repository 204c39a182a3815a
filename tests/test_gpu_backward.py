"""GPU parity of the layer backward (dX, every weight gradient, dlogits, dW_router) against the
float64 oracle with the GPU's own top-k selection, through the C ABI; plus run-to-run bit
identity of every gradient."""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, LayerShape, make_layer
from tests._helpers import assert_close, dims_of, ensure_lib, f64, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": WORKLOADS["tiny"].with_(backward=True),
    "ragged_skew": LayerShape("ragged_skew", 300, 384, 16, 4, 256, 384, 1, 0.0, "zipf", "bf16", True, 21),
    "noshared": LayerShape("noshared", 190, 256, 8, 3, 128, 0, 0, 0.05, "normal0.1", "bf16", True, 22),
    # 256-column weight-gradient tiles (d, F, Fs multiples of 256) with several M and N tiles
    # per problem; skewed routing leaves experts with few or no rows
    "wide_tiles_skew": LayerShape("wide_tiles_skew", 260, 512, 8, 2, 512, 512, 1, 0.0, "zipf", "bf16", True, 23),
    "wide_tiles_noshared": LayerShape("wide_tiles_noshared", 200, 256, 8, 3, 256, 0, 0, 0.0, "zipf", "bf16", True, 24),
    # training forward in CTA pairs (at least 320 routed rows per expert)
    "pairs_train": LayerShape("pairs_train", 880, 256, 8, 3, 256, 256, 1, 0.0, "zipf", "bf16", True, 25),
    # the largest expert count and top-k the ABI accepts (E = 512, k = 8): the router GEMM's
    # N = 512 and dW_router's two 256-column tiles
    "max_E_k": LayerShape("max_E_k", 200, 256, 512, 8, 256, 256, 1, 0.0, "normal0.1", "bf16", True, 26),
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_parity_and_determinism(name):
    ensure_lib()
    shape = CASES[name]
    L = make_layer(shape, "cpu", with_dy=True)
    Ld = to_dev(L)
    D = dims_of(shape)
    layer = mok.MoELayer(D, Ld)
    layer.forward(Ld["x"], training=True)
    g = layer.backward(Ld["x"], Ld["dY"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0 and mok.read_status(layer._ws_bwd) == 0

    idx = layer.routing["topk_idx"].cpu().numpy()
    x, Wr = f64(L["x"]), f64(L["W_router"])
    b = None if L["bias"] is None else f64(L["bias"])
    logits = oracle.router_logits(x, Wr, b)
    shared = None if not shape.n_shared else (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))
    ref = oracle.moe_backward(x, f64(L["dY"]), Wr, f64(L["W_gate"]), f64(L["W_up"]),
                              f64(L["W_down"]), shared, logits, idx)
    for key in ("dX", "dW_gate", "dW_up", "dW_down", "dlogits", "dW_router"):
        assert_close(key, f64(g[key]), ref[key])
    if shape.n_shared:
        for key in ("dWs_gate", "dWs_up", "dWs_down"):
            assert_close(key, f64(g[key]), ref[key])
    # experts without tokens get exact zeros
    empty = np.nonzero(np.bincount(idx.ravel(), minlength=shape.E) == 0)[0]
    for e in empty:
        assert not g["dW_gate"][e].any() and not g["dW_down"][e].any()

    g2 = layer.backward(Ld["x"], Ld["dY"])
    torch.cuda.synchronize()
    for key, v in g.items():
        if v is not None:
            assert torch.equal(v, g2[key]), key
