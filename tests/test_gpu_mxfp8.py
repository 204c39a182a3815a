"""GPU parity of the MXFP8 path through the C ABI.

* Quantiser (mok_mx_quantize_rows) and prepared weights (mok_prepare_weights): bit-exact codes
  and scale bytes against the oracle's quantiser on the same bf16 values.
* Forward: within max|d| <= 6e-2 max|ref| (and a mean relative error <= 1e-2) of the oracle's
  MXFP8 reading, which quantises x, the weights and h exactly where the method does and computes
  in float64; bit-identical reruns.  The distance to the unquantised float64 layer is reported
  and bounded by the oracle's own MXFP8-vs-float64 distance plus 1e-2: E4M3 rounding of random-
  sign products does not average out relative to the output (about 6-7% on these inputs even in
  float64).
"""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, LayerShape, make_layer
from tests._helpers import LazyExperts, assert_close, dims_of, ensure_lib, errors, f64, to_dev

pytestmark = pytest.mark.gpu

MX_MAX_REL = 6e-2


def _edge_rows():
    rng = np.random.default_rng(0)
    a = (rng.standard_normal((64, 256)) * np.logspace(-6, 4, 64)[:, None]).astype(np.float32)
    a[0, :32] = 0.0                                   # all-zero block
    a[1, :32] = 448.0                                 # amax exactly 448 * 2^0
    a[2, 32:64] = 448.0 * 2.0 ** -5                   # amax exactly 448 * 2^-5
    a[3, :] = np.float32(1e-30)                       # tiny
    a[4, 5] = -3.0e4                                  # one large value in a block
    a[5, :] = np.float32(2.0 ** -130)                 # subnormal bf16 values
    return torch.from_numpy(a).to(torch.bfloat16)


def test_quantizer_bit_exact():
    ensure_lib()
    src = _edge_rows()
    q, sc = mok.mx_quantize_rows(src.cuda())
    torch.cuda.synchronize()
    q_ref, sc_ref = oracle.mx_quantize(f64(src))
    assert (sc.cpu().numpy() == sc_ref).all()
    assert (q.cpu().numpy() == q_ref).all()


def _mx_shape(base, **kw):
    return base.with_(dtype="mxfp8", **kw)


def scales_from_atoms(flat, n, N, K):
    """[n][N][K/32] scale bytes from the 512-byte atoms [n][N/128][K/128] of mok.h: row
    128a + 32 r1 + r0, block 4b + j at byte 16 r0 + 4 r1 + j of atom (a, b)."""
    a = flat.reshape(n, N // 128, K // 128, 32, 4, 4)          # [n][a][b][r0][r1][j]
    return a.transpose(0, 1, 4, 3, 2, 5).reshape(n, N, K // 32)  # [n][a][r1][r0][b][j]


def test_atom_reader_on_a_known_layout():
    """The atom reader places the byte written for (row, block) by the rule in mok.h back at
    (row, block) (a layout check of the test's own reader, no GPU work)."""
    n, N, K = 2, 256, 512
    flat = np.zeros(n * N * K // 32, dtype=np.int64)
    for m in range(n):
        for row in range(N):
            for blk in range(K // 32):
                a, r = divmod(row, 128)
                b, j = divmod(blk, 4)
                off = ((m * (N // 128) + a) * (K // 128) + b) * 512 + 16 * (r % 32) + 4 * (r // 32) + j
                flat[off] = (m * N + row) * 1000 + blk
    got = scales_from_atoms(flat, n, N, K)
    want = (np.arange(n)[:, None, None] * N + np.arange(N)[None, :, None]) * 1000 + np.arange(K // 32)
    assert (got == want).all()


def test_prepared_weights_bit_exact():
    ensure_lib()
    shape = _mx_shape(WORKLOADS["tiny"], F=256, F_shared=128)
    L = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape, dtype=mok.MOK_MXFP8)
    prep = mok.prepare_weights(D, L)
    torch.cuda.synchronize()
    buf = prep.cpu().numpy()
    E, d, F, Fs = shape.E, shape.d, shape.F, shape.F_shared

    def al(n):
        return (n + 1023) // 1024 * 1024

    sizes = [E * F * d, E * F * d // 32, E * F * d, E * F * d // 32, E * d * F, E * d * F // 32,
             Fs * d, Fs * d // 32, Fs * d, Fs * d // 32, d * Fs, d * Fs // 32]
    offs = np.cumsum([0] + [al(n) for n in sizes])
    mats = [(L["W_gate"], E, d, F), (L["W_up"], E, d, F), (L["W_down"], E, F, d),
            (L["Ws_gate"][None], 1, d, Fs), (L["Ws_up"][None], 1, d, Fs), (L["Ws_down"][None], 1, Fs, d)]
    for i, (W, n, K, N) in enumerate(mats):
        Wt = np.swapaxes(f64(W), 1, 2)               # [n][N][K]: K-major
        q_ref, s_ref = oracle.mx_quantize(Wt)
        q = buf[offs[2 * i]:offs[2 * i] + n * N * K].reshape(n, N, K)
        s = scales_from_atoms(buf[offs[2 * i + 1]:offs[2 * i + 1] + n * N * K // 32], n, N, K)
        assert (s == s_ref).all(), f"scales of matrix {i}"
        assert (q == q_ref).all(), f"codes of matrix {i}"


CASES = {
    "tiny_mx": _mx_shape(WORKLOADS["tiny"]),
    "ragged_mx": LayerShape("ragged_mx", 300, 512, 16, 4, 256, 384, 1, 0.0, "zipf", "mxfp8", False, 31),
    "noshared_mx": LayerShape("noshared_mx", 130, 256, 8, 8, 128, 0, 0, 0.05, "none", "mxfp8", False, 32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_mxfp8_forward_parity(name):
    ensure_lib()
    shape = CASES[name]
    L = make_layer(shape, "cpu")
    Ld = to_dev(L)
    D = dims_of(shape, dtype=mok.MOK_MXFP8)
    Ld["prepared"] = mok.prepare_weights(D, Ld)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, Ld["x"], Ld["W_router"], Ld["bias"], ws)
    r = mok.dispatch_index(D, idx, w, ws)
    y = mok.moe_forward(D, Ld, Ld["x"], r, ws)
    y2 = mok.moe_forward(D, Ld, Ld["x"], r, ws)
    torch.cuda.synchronize()
    assert mok.read_status(ws) == 0
    assert torch.equal(y, y2)
    x = f64(L["x"])
    b = None if L["bias"] is None else f64(L["bias"])
    got = idx.cpu().numpy()
    wr = oracle.weights_for_selection(oracle.router_logits(x, f64(L["W_router"]), b), got)
    sh = None if not shape.n_shared else (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))
    Wg, Wu, Wd = f64(L["W_gate"]), f64(L["W_up"]), f64(L["W_down"])
    y_ref = oracle.moe_forward(x, Wg, Wu, Wd, sh, got, wr)
    y_mx = oracle.moe_forward_mxfp8(x, Wg, Wu, Wd, sh, got, wr)
    mx, mn = assert_close("y vs MXFP8 reading", f64(y), y_mx, max_rel=MX_MAX_REL, mean_rel=1e-2)
    own_mx, own_mn = errors(y_mx, y_ref)
    mx2, mn2 = assert_close("y vs float64", f64(y), y_ref, max_rel=own_mx + 1e-2, mean_rel=own_mn + 1e-2)
    print(f"{name}: vs MXFP8 reading max_rel {mx:.2e} mean_rel {mn:.2e}; vs float64 {mx2:.2e} "
          f"{mn2:.2e} (oracle MXFP8 vs float64 {own_mx:.2e} {own_mn:.2e})")


def test_fullsize_mxfp8_forward_sampled():
    ensure_lib()
    shape = WORKLOADS["dsv3_mxfp8_fwd"]
    L = make_layer(shape, "cuda")
    D = dims_of(shape, dtype=mok.MOK_MXFP8)
    L["prepared"] = mok.prepare_weights(D, L)
    layer = mok.MoELayer(D, L)
    y = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0
    got = layer.routing["topk_idx"].cpu().numpy()
    toks = [shape.T - 1]
    x = f64(L["x"][toks])
    wr = oracle.weights_for_selection(oracle.router_logits(x, f64(L["W_router"]), f64(L["bias"])), got[toks])
    sh = (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))
    Wg, Wu, Wd = LazyExperts(L["W_gate"]), LazyExperts(L["W_up"]), LazyExperts(L["W_down"])
    y_mx = oracle.moe_forward_mxfp8(x, Wg, Wu, Wd, sh, got[toks], wr)
    assert_close("y sampled vs MXFP8 reading", f64(y[toks]), y_mx, max_rel=MX_MAX_REL, mean_rel=1e-2)
