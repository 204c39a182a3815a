"""GPU parity of the router, the pull schedule and the layer forward against the float64 oracle,
through the C ABI.  Sizes span several 128-row tiles with ragged tails, empty experts, a hot
expert, k = E, no shared expert, F != Fs and d not a multiple of 256."""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, LayerShape, make_layer
from tests._helpers import NEAR_TIE, assert_close, dims_of, ensure_lib, f64, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": WORKLOADS["tiny"],
    "ragged_skew": LayerShape("ragged_skew", 300, 384, 16, 4, 256, 384, 1, 0.0, "zipf", "bf16", False, 11),
    "k_eq_E_noshared": LayerShape("k_eq_E_noshared", 129, 256, 8, 8, 128, 0, 0, 0.05, "none", "bf16", False, 12),
    "one_token": LayerShape("one_token", 1, 256, 16, 3, 256, 128, 1, 0.0, "normal0.1", "bf16", False, 13),
    "wide_E": LayerShape("wide_E", 200, 256, 384, 8, 128, 128, 1, 0.0, "normal0.1", "bf16", False, 14),
    # at least 320 routed rows per expert: gate/up and down in CTA pairs of 256-row tiles, skewed
    # so that experts span several pair tiles, end mid-tile or hold no rows
    "pairs": LayerShape("pairs", 720, 256, 8, 4, 256, 256, 1, 0.0, "zipf", "bf16", False, 15),
    # pairs with a Kimi-like tail: 19 of 32 experts hold at most 128 rows (1 to 109; several at
    # most 64, so the second CTA of their M = 128 pair tile has no row) beside experts of up to
    # 2500 rows in many 256-row pair tiles
    "pairs_tail": LayerShape("pairs_tail", 2600, 256, 32, 4, 256, 256, 1, 0.0, "zipf", "bf16", False, 20),
    # pairs for gate/up only (d not a multiple of 256: 128-column down tiles without pairs)
    "pairs_gu_only": LayerShape("pairs_gu_only", 660, 384, 8, 4, 128, 0, 0, 0.0, "normal0.1", "bf16", False, 16),
    # the largest expert count and top-k the ABI accepts (E = 512, k = 8)
    "max_E_k": LayerShape("max_E_k", 300, 256, 512, 8, 128, 128, 1, 0.0, "normal0.1", "bf16", False, 17),
}


def _oracle_inputs(L):
    return dict(
        x=f64(L["x"]), Wr=f64(L["W_router"]),
        b=None if L["bias"] is None else f64(L["bias"]),
        Wg=f64(L["W_gate"]), Wu=f64(L["W_up"]), Wd=f64(L["W_down"]),
        shared=None if L["Ws_gate"] is None else (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"])),
    )


def _run_gpu(shape, L):
    D = dims_of(shape)
    Ld = to_dev(L)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, logits = mok.route(D, Ld["x"], Ld["W_router"], Ld["bias"], ws, want_logits=True)
    routing = mok.dispatch_index(D, idx, w, ws)
    y = mok.moe_forward(D, Ld, Ld["x"], routing, ws)
    torch.cuda.synchronize()
    assert mok.read_status(ws) == 0
    return D, Ld, ws, idx, w, logits, routing, y


def check_route(shape, O, idx, w, logits):
    l64, l32, idx_ref, _ = oracle.route(O["x"], O["Wr"], O["b"], shape.k)
    got_idx = idx.cpu().numpy()
    gap = oracle.topk_gap(l32, shape.k)
    ok = gap >= NEAR_TIE
    # selection: bit-exact on every token without a near tie at the k-th place
    assert (np.sort(got_idx[ok], axis=1) == np.sort(idx_ref[ok], axis=1)).all()
    # slot order: descending logit, checked where the selected logits are not near-equal
    top = -np.sort(-l32.astype(np.float64), axis=1)[:, : shape.k]
    ordered = ok
    if shape.k > 1:
        ordered = ok & ((top[:, :-1] - top[:, 1:]).min(axis=1) >= NEAR_TIE)
    assert (got_idx[ordered] == idx_ref[ordered]).all()
    # logits of the tensor-core router GEMM vs the float64 definition
    assert_close("logits", logits.cpu().numpy(), l64, max_rel=1e-4, mean_rel=1e-5)
    # weights at the GPU's own selection (softmax renormalised over the selection): since
    # d log w_j = dl_j - sum_i w_i dl_i, each token's weights sit within 2 max_j |dl_j| (its
    # selected logits' error against float64) relative, plus fp32 rounding of the softmax
    w_ref = oracle.weights_for_selection(l64, got_idx)
    sel = np.take_along_axis(logits.cpu().numpy().astype(np.float64) - l64, got_idx.astype(np.int64), axis=1)
    bound = (2.0 * np.abs(sel).max(axis=1, keepdims=True) + 4e-6) * w_ref + 1e-7
    assert (np.abs(w.cpu().numpy() - w_ref) <= bound).all()
    return l64, got_idx, int((~ok).sum())


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


@pytest.mark.parametrize("name", list(CASES))
def test_route_dispatch_forward_parity(name):
    shape = CASES[name]
    L = make_layer(shape, "cpu")
    O = _oracle_inputs(L)
    D, Ld, ws, idx, w, logits, routing, y = _run_gpu(shape, L)
    l64, got_idx, n_near = check_route(shape, O, idx, w, logits)

    # pull schedule: bit-exact against the oracle's scan on the GPU's selection
    counts, offsets, sorted_tok, inv_pos = oracle.dispatch(got_idx, shape.E)
    assert (routing["counts"].cpu().numpy() == counts).all()
    assert (routing["offsets"].cpu().numpy() == offsets).all()
    assert (routing["sorted_tok"].cpu().numpy() == sorted_tok).all()
    assert (routing["inv_pos"].cpu().numpy() == inv_pos).all()
    sw_ref = w.cpu().numpy().reshape(-1)[np.argsort(inv_pos.reshape(-1))]
    assert (routing["sorted_w"].cpu().numpy() == sw_ref).all()

    # layer output with the GPU's selection and the oracle's weights
    w_ref = oracle.weights_for_selection(l64, got_idx)
    y_ref = oracle.moe_forward(O["x"], O["Wg"], O["Wu"], O["Wd"], O["shared"], got_idx, w_ref)
    assert_close("y", f64(y), y_ref)

    # bit-identical on a second run
    y2 = mok.moe_forward(D, Ld, Ld["x"], routing, ws)
    idx2, w2, _ = mok.route(D, Ld["x"], Ld["W_router"], Ld["bias"], ws)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(idx, idx2) and torch.equal(w, w2)


def test_worked_pull_example_on_gpu():
    """Page "Метод и эксперименты": E2 <- [0,2,9,15], E5 <- [3,8], E7 <- [1,4,5,6]."""
    ensure_lib()
    route = {0: 2, 1: 7, 2: 2, 3: 5, 4: 7, 5: 7, 6: 7, 7: 0, 8: 5, 9: 2, 10: 0, 11: 0, 12: 0,
             13: 0, 14: 0, 15: 2}
    D = mok.dims(16, 128, 8, 1, 128, 0, 0)
    idx = torch.tensor([[route[t]] for t in range(16)], dtype=torch.int32, device="cuda")
    w = torch.ones((16, 1), dtype=torch.float32, device="cuda")
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    r = mok.dispatch_index(D, idx, w, ws)
    off = r["offsets"].cpu().tolist()
    tok = r["sorted_tok"].cpu().tolist()
    assert tok[off[2]:off[3]] == [0, 2, 9, 15]
    assert tok[off[5]:off[6]] == [3, 8]
    assert tok[off[7]:off[8]] == [1, 4, 5, 6]
    assert mok.read_status(ws) == 0


def test_out_of_range_expert_index_sets_status():
    ensure_lib()
    D = mok.dims(8, 128, 8, 2, 128, 0, 0)
    idx = torch.tensor([[0, 1]] * 7 + [[3, 99]], dtype=torch.int32, device="cuda")
    w = torch.full((8, 2), 0.5, dtype=torch.float32, device="cuda")
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    r = mok.dispatch_index(D, idx, w, ws)
    assert mok.read_status(ws) == -6
    assert r["offsets"].cpu().tolist()[-1] == 15       # the bad route is dropped
    assert r["inv_pos"].cpu()[7, 1].item() == -1
    mok.clear_status(ws)
    assert mok.read_status(ws) == 0


def test_zero_tokens_is_a_no_op():
    ensure_lib()
    shape = CASES["tiny"].with_(T=0)
    D = dims_of(shape)
    L = to_dev(make_layer(CASES["tiny"], "cpu"))
    x = torch.empty((0, shape.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, x, L["W_router"], L["bias"], ws)
    r = mok.dispatch_index(D, idx, w, ws)
    y = mok.moe_forward(D, L, x, r, ws)
    torch.cuda.synchronize()
    assert y.shape == (0, shape.d) and r["offsets"].cpu().tolist() == [0] * (shape.E + 1)


def test_host_buffer_entry_point_matches_device_path():
    ensure_lib()
    shape = CASES["tiny"]
    L = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, L["x"], L["W_router"], L["bias"], ws)
    y_dev = mok.moe_forward(D, L, L["x"], mok.dispatch_index(D, idx, w, ws), ws)
    wsh = torch.zeros(mok.workspace_size(D) + mok.host_extra_size(D), dtype=torch.uint8, device="cuda")
    xh = L["x"].cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    mok.layer_forward_host(D, L, xh, yh, wsh)
    torch.cuda.synchronize()
    assert torch.equal(yh, y_dev.cpu())


def test_host_entry_point_back_to_back_calls():
    """Three host-buffer calls on one workspace with no synchronisation between them: each call's
    copy of x goes to one of two device buffers in turn, so the third reuses the first one's
    buffer while the layer may still run; every y must match its own device-path forward."""
    ensure_lib()
    shape = CASES["ragged_skew"]
    L = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape)
    xs = [L["x"], (L["x"].float() * 0.5).to(torch.bfloat16), -L["x"]]
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    y_dev = []
    for x in xs:
        idx, w, _ = mok.route(D, x, L["W_router"], L["bias"], ws)
        y_dev.append(mok.moe_forward(D, L, x, mok.dispatch_index(D, idx, w, ws), ws).cpu())
    torch.cuda.synchronize()
    wsh = torch.zeros(mok.workspace_size(D) + mok.host_extra_size(D), dtype=torch.uint8, device="cuda")
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.empty_like(h).pin_memory() for h in xh]
    for xi, yi in zip(xh, yh):
        mok.layer_forward_host(D, L, xi, yi, wsh)
    torch.cuda.synchronize()
    assert mok.read_status(wsh) == 0
    for i in range(3):
        assert torch.equal(yh[i], y_dev[i]), i


def test_host_entry_point_pageable_output():
    """y_host in pageable memory: the layer combines into the workspace and copies y back (the
    pinned case writes y straight into host memory); both give the device path's bytes."""
    ensure_lib()
    shape = CASES["tiny"]
    L = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, L["x"], L["W_router"], L["bias"], ws)
    y_dev = mok.moe_forward(D, L, L["x"], mok.dispatch_index(D, idx, w, ws), ws).cpu()
    wsh = torch.zeros(mok.workspace_size(D) + mok.host_extra_size(D), dtype=torch.uint8, device="cuda")
    xh = L["x"].cpu().pin_memory()
    yh = torch.empty_like(xh)          # pageable
    assert not yh.is_pinned()
    mok.layer_forward_host(D, L, xh, yh, wsh)
    torch.cuda.synchronize()
    assert torch.equal(yh, y_dev)


def test_layer_is_cuda_graph_capturable():
    """The entry points allocate nothing, synchronise nothing and take their stream from the
    caller, so a whole training step (route, pull schedule, forward, backward) can be captured in
    a CUDA graph and replayed: replays give the eager results bit for bit, also after new inputs
    are copied into the captured buffers."""
    ensure_lib()
    shape = CASES["ragged_skew"].with_(backward=True)
    L = to_dev(make_layer(shape, "cpu", with_dy=True))
    D = dims_of(shape)
    layer = mok.MoELayer(D, L)
    x = L["x"].clone()
    dY = L["dY"].clone()

    def step():
        y = layer.forward(x, training=True)
        g = layer.backward(x, dY)
        return y, g

    y0, g0 = step()                      # eager: also sets up the backward workspace
    y0, g0 = y0.clone(), {k: (v.clone() if v is not None else None) for k, v in g0.items()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y, g = step()
    graph.replay()
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0 and mok.read_status(layer._ws_bwd) == 0
    assert torch.equal(y, y0)
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(g[k], v), k
    # new inputs through the captured buffers
    x2 = make_layer(shape.with_(cid=shape.cid + 100), "cpu", with_dy=True)
    x.copy_(x2["x"].cuda())
    dY.copy_(x2["dY"].cuda())
    graph.replay()
    torch.cuda.synchronize()
    y_replay, dX_replay = y.clone(), g["dX"].clone()
    y_eager, g_eager = step()
    torch.cuda.synchronize()
    assert torch.equal(y_replay, y_eager)
    assert torch.equal(dX_replay, g_eager["dX"])


@pytest.mark.parametrize("name", ["tiny", "k_eq_E_noshared", "one_token", "wide_E", "max_E_k"])
def test_fused_schedule_is_bit_identical(name):
    """The fused schedule (gate/up and down in one persistent launch, tiles claimed from a device
    work counter, down tiles gated by per-M-tile readiness counters) gives exactly the output of
    the two-launch schedule, twice in a row."""
    shape = CASES[name]
    L = make_layer(shape, "cpu")
    D, Ld, ws, idx, w, logits, routing, y0 = _run_gpu(shape, L)
    prev = mok.set_forward_schedule(mok.SCHEDULE_FUSED)
    try:
        y1 = mok.moe_forward(D, Ld, Ld["x"], routing, ws)
        y2 = mok.moe_forward(D, Ld, Ld["x"], routing, ws)
        torch.cuda.synchronize()
    finally:
        mok.set_forward_schedule(prev)
    assert mok.read_status(ws) == 0
    assert torch.equal(y1, y0) and torch.equal(y2, y0)
