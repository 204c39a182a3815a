"""GPU parity of the NVFP4 variant through the C ABI.

* Prepared weights (mok_prepare_weights with MOK_NVFP4): bit-exact codes, scale bytes and
  per-matrix decode scales against the oracle's quantiser (oracle/nvfp4.py) on the same bf16
  values, read back through the layout include/mok.h documents.
* Forward: within max|d| <= 2e-2 max|ref| (mean 5e-3) of the oracle's NVFP4 reading (the
  quantisation points of the path, the same calibrated activation amaxes, float64 sums); the
  cases cover ragged experts, no shared expert, and calibrated amaxes below the data (values
  saturate); bit-identical reruns.  The full NVFP4 forward workloads (E=256 at T=4096, and the
  T=64 decode) on at least 64 tokens that reach every active expert.
* The distance to the unquantised float64 layer is reported: NVFP4 keeps about three
  significant bits per element, so it is several per cent, and the oracle's own distance bounds
  the GPU's.
"""

import numpy as np
import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
import oracle
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, LayerShape, make_layer
from tests._fullsize import experts_of, oracle_pool, sampled_tokens
from tests._helpers import assert_close, dims_of, ensure_lib, errors, f64, to_dev

pytestmark = pytest.mark.gpu

# h codes differ where the GPU's fp32 h and the oracle's float64 h straddle an E2M1 rounding
# point; the bf16 output rounding adds 2^-9.  Bars: the bf16 ones.
NV_MAX_REL = 2e-2
NV_MEAN_REL = 5e-3
AMAX_H = 8.0   # calibrated amax of h for these N(0, 1) inputs (a few values beyond it saturate)


def _al(n):
    return (n + 1023) // 1024 * 1024


def prepared_regions(buf, E, d, F, Fs):
    """The regions of an NVFP4 prepared buffer, in the order and 1 KB alignment of mok.h."""
    mats = [(E, d, F), (E, d, F), (E, F, d), (1, d, Fs), (1, d, Fs), (1, Fs, d)]
    sizes = []
    for n, K, N in mats:
        sizes += [n * K * N // 2, n * K * N // 16]
    nmat = 3 * E + 3
    sizes += [4 * nmat, 4 * nmat, 8]
    offs = np.cumsum([0] + [_al(n) for n in sizes])
    out = []
    for i, (n, K, N) in enumerate(mats):
        q = buf[offs[2 * i]:offs[2 * i] + n * K * N // 2].reshape(n, K // 64, N, 32)
        codes = np.empty((n, K // 64, N, 64), dtype=np.uint8)
        codes[..., 0::2] = q & 0xF
        codes[..., 1::2] = q >> 4
        codes = codes.transpose(0, 2, 1, 3).reshape(n, N, K)              # [n][N][K]
        s = buf[offs[2 * i + 1]:offs[2 * i + 1] + n * K * N // 16].reshape(n, K // 64, N, 4)
        scales = s.transpose(0, 2, 1, 3).reshape(n, N, K // 16)            # [n][N][K/16]
        out.append((codes, scales))
    g = buf[offs[12]:offs[12] + 4 * nmat].view(np.float32)
    act = buf[offs[14]:offs[14] + 8].view(np.float32)
    return out, g, act


def test_prepared_weights_bit_exact():
    ensure_lib()
    shape = WORKLOADS["tiny"].with_(dtype="nvfp4", F=256, F_shared=128)
    L = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape, dtype=mok.MOK_NVFP4)
    prep = mok.prepare_weights(D, L)
    mok.nvfp4_set_activation_amax(D, prep, 3.0, 5.0)
    torch.cuda.synchronize()
    E, d, F, Fs = shape.E, shape.d, shape.F, shape.F_shared
    regions, g, act = prepared_regions(prep.cpu().numpy(), E, d, F, Fs)
    mats = [f64(L["W_gate"]), f64(L["W_up"]), f64(L["W_down"]), f64(L["Ws_gate"])[None],
            f64(L["Ws_up"])[None], f64(L["Ws_down"])[None]]
    g_idx = [np.arange(E), E + np.arange(E), 2 * E + np.arange(E), [3 * E], [3 * E + 1], [3 * E + 2]]
    for i, W in enumerate(mats):
        codes, scales = regions[i]
        for m in range(W.shape[0]):
            q_ref, s_ref, g_ref = oracle.nv_quantize(W[m].T)              # [N][K] along K
            assert (scales[m] == s_ref).all(), f"scales of matrix {i}.{m}"
            assert (codes[m] == q_ref).all(), f"codes of matrix {i}.{m}"
            assert g[g_idx[i][m]] == g_ref, f"decode scale of matrix {i}.{m}"
    assert act.tolist() == [3.0, 5.0]


CASES = {
    "tiny_nv": (WORKLOADS["tiny"].with_(name="tiny_nv", dtype="nvfp4"), None),
    "ragged_nv": (LayerShape("ragged_nv", 300, 512, 16, 4, 256, 384, 1, 0.0, "zipf", "nvfp4", False, 33), None),
    "noshared_nv": (LayerShape("noshared_nv", 130, 256, 8, 8, 128, 0, 0, 0.05, "none", "nvfp4", False, 34), None),
    # calibrated amaxes below the data: x values above half its amax and h values above 1 saturate
    "clip_nv": (LayerShape("clip_nv", 200, 256, 8, 2, 256, 256, 1, 0.0, "normal0.1", "nvfp4", False, 35), (0.5, 1.0)),
    # about 32 rows per expert: tiles on both sides of the 32-row A boxes
    "rows32_nv": (LayerShape("rows32_nv", 128, 256, 8, 2, 256, 128, 1, 0.0, "none", "nvfp4", False, 36), None),
    # fewer tokens than a 32-row box: the shared expert's tile takes it too
    "t24_nv": (LayerShape("t24_nv", 24, 512, 16, 4, 128, 256, 1, 0.0, "normal0.1", "nvfp4", False, 37), None),
}


def _amaxes(x, clip):
    ax = float(np.abs(x).max())
    return (ax, AMAX_H) if clip is None else (clip[0] * ax, clip[1])


@pytest.mark.parametrize("name", list(CASES))
def test_nvfp4_forward_parity(name):
    ensure_lib()
    shape, clip = CASES[name]
    L = make_layer(shape, "cpu")
    Ld = to_dev(L)
    D = dims_of(shape, dtype=mok.MOK_NVFP4)
    x = f64(L["x"])
    amax_x, amax_h = _amaxes(x, clip)
    Ld["prepared"] = mok.prepare_weights(D, Ld)
    mok.nvfp4_set_activation_amax(D, Ld["prepared"], amax_x, amax_h)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, Ld["x"], Ld["W_router"], Ld["bias"], ws)
    r = mok.dispatch_index(D, idx, w, ws)
    y = mok.moe_forward(D, Ld, Ld["x"], r, ws)
    y2 = mok.moe_forward(D, Ld, Ld["x"], r, ws)
    torch.cuda.synchronize()
    assert mok.read_status(ws) == 0
    assert torch.equal(y, y2)
    b = None if L["bias"] is None else f64(L["bias"])
    got = idx.cpu().numpy()
    wr = oracle.weights_for_selection(oracle.router_logits(x, f64(L["W_router"]), b), got)
    sh = None if not shape.n_shared else (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))
    Wg, Wu, Wd = f64(L["W_gate"]), f64(L["W_up"]), f64(L["W_down"])
    y_nv = oracle.moe_forward_nvfp4(x, Wg, Wu, Wd, sh, got, wr, np.float32(amax_x), amax_h)
    y_ref = oracle.moe_forward(x, Wg, Wu, Wd, sh, got, wr)
    yg = f64(y)
    mx, mn = assert_close("y vs NVFP4 reading", yg, y_nv, max_rel=NV_MAX_REL, mean_rel=NV_MEAN_REL)
    own_mx, own_mn = errors(y_nv, y_ref)
    mx2, mn2 = assert_close("y vs float64", yg, y_ref, max_rel=own_mx + 1e-2, mean_rel=own_mn + 1e-2)
    print(f"{name}: vs NVFP4 reading max_rel {mx:.2e} mean_rel {mn:.2e}; vs float64 {mx2:.2e} "
          f"{mn2:.2e} (oracle NVFP4 vs float64 {own_mx:.2e} {own_mn:.2e})")


def test_nvfp4_rejects_training_and_bad_calibration():
    ensure_lib()
    shape = WORKLOADS["tiny"].with_(dtype="nvfp4")
    Ld = to_dev(make_layer(shape, "cpu"))
    D = dims_of(shape, dtype=mok.MOK_NVFP4)
    Ld["prepared"] = mok.prepare_weights(D, Ld)
    assert mok.saved_size(D) == 0
    for bad in ((-1.0, 1.0), (1.0, float("nan")), (float("inf"), 1.0)):
        with pytest.raises(mok.MokError):
            mok.nvfp4_set_activation_amax(D, Ld["prepared"], *bad)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    idx, w, _ = mok.route(D, Ld["x"], Ld["W_router"], Ld["bias"], ws)
    r = mok.dispatch_index(D, idx, w, ws)
    fake_saved = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(mok.MokError):
        mok.moe_forward(D, Ld, Ld["x"], r, ws, saved=fake_saved)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["dsv3_nvfp4_fwd", "dsv3_nvfp4_decode_t64"])
def test_fullsize_nvfp4_forward_sampled(name):
    """The NVFP4 forward workloads at full size (E=256; T=4096, and T=64, where every expert
    tile holds at most 32 rows and loads them through the 32-row maps): y on at least 64 tokens
    that reach every active expert (every token at T=64), against the oracle's NVFP4 reading
    (one expert per pool job)."""
    ensure_lib()
    shape = WORKLOADS[name]
    L = make_layer(shape, "cuda")
    D = dims_of(shape, dtype=mok.MOK_NVFP4)
    L["prepared"] = mok.prepare_weights(D, L)
    amax_x = float(L["x"].abs().max())
    mok.nvfp4_set_activation_amax(D, L["prepared"], amax_x, AMAX_H)
    layer = mok.MoELayer(D, L)
    y = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert mok.read_status(layer.ws) == 0
    got = layer.routing["topk_idx"].cpu().numpy()
    counts = np.bincount(got.ravel(), minlength=shape.E)
    toks = sampled_tokens(got, counts, shape.T)
    x = f64(L["x"][toks])
    wr = oracle.weights_for_selection(oracle.router_logits(x, f64(L["W_router"]), f64(L["bias"])), got[toks])
    sh = (f64(L["Ws_gate"]), f64(L["Ws_up"]), f64(L["Ws_down"]))
    Wg, Wu, Wd = experts_of(L)
    with oracle_pool() as pmap:
        y_nv = oracle.moe_forward_nvfp4(x, Wg, Wu, Wd, sh, got[toks], wr, np.float32(amax_x), AMAX_H,
                                        expert_map=pmap)
    mx, mn = assert_close("y sampled vs NVFP4 reading", f64(y[toks]), y_nv, max_rel=NV_MAX_REL,
                          mean_rel=NV_MEAN_REL)
    print(f"{name}: {len(toks)} tokens reaching {(counts > 0).sum()} experts: vs NVFP4 "
          f"reading max_rel {mx:.2e} mean_rel {mn:.2e}")
