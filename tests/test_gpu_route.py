"""The router alone at the full workload sizes (x and W_router only on the device), against the
float64 oracle: selection bit-exact on every token off near ties, slot order, logits and weights.
The token tiles times the K splits fill the GPU once, so these sizes run the cluster form of the
router (2 to 8 K-split CTAs per token tile reducing their partial logits through distributed
shared memory) as well as the one-split form (the Kimi-class batch); E = 384 and E = 512 reduce
the logits in column chunks.  The same call is the small profiling command of the router."""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, LayerShape, make_layer
from tests._helpers import dims_of, ensure_lib, f64
from tests.test_gpu_forward import check_route

pytestmark = pytest.mark.gpu

ROUTE_CASES = {
    "dsv3_bf16_fwd": WORKLOADS["dsv3_bf16_fwd"],             # T = 4096: 4 splits
    "dsv3_bf16_train": WORKLOADS["dsv3_bf16_train"],         # T = 8192: 2 splits
    "kimi_skew_bf16_fwd": WORKLOADS["kimi_skew_bf16_fwd"],   # T = 16384: one split, E = 384
    "dsv3_decode_t64": WORKLOADS["dsv3_decode_t64"],         # T = 64: 8 splits
    "wide_E_512": LayerShape("wide_E_512", 4000, 7168, 512, 8, 2048, 2048, 1, 0.0, "normal0.1",
                             "bf16", False, 18),            # 4 splits, two column chunks
    # 39 token tiles (2 splits), E = 128: one 128-column MMA per tile
    "odd_tiles_E128": LayerShape("odd_tiles_E128", 4992, 7168, 128, 8, 2048, 2048, 1, 0.0,
                                 "normal0.1", "bf16", False, 19),
}


def _router_inputs(shape):
    """x, W_router and the bias of the workload, drawn on the GPU with the workload's seeds
    (the expert weights are not needed)."""
    L = make_layer(shape.with_(E=shape.E, F=128, F_shared=128, d=shape.d), "cuda")
    return L["x"], L["W_router"], L["bias"]


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_route_fullsize(name):
    ensure_lib()
    shape = ROUTE_CASES[name]
    x, Wr, b = _router_inputs(shape)
    D = dims_of(shape)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, logits = mok.route(D, x, Wr, b, ws, want_logits=True)
    idx2, w2, _ = mok.route(D, x, Wr, b, ws)
    torch.cuda.synchronize()
    assert mok.read_status(ws) == 0
    assert torch.equal(idx, idx2) and torch.equal(w, w2)      # bit-identical reruns
    O = {"x": f64(x), "Wr": f64(Wr), "b": None if b is None else f64(b)}
    _, got, n_near = check_route(shape, O, idx, w, logits)
    print(f"{name}: {n_near} near-tie tokens excluded of {shape.T}")
