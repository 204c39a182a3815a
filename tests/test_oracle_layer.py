"""Pins of the oracle's SwiGLU expert FFN, layer forward and backward, on the CPU.

* SiLU at closed-form points.
* The FFN with (scaled) permutation-matrix weights, whose output is known elementwise.
* Layer invariants: k = E with identical experts gives shared + FFN; permuting tokens permutes the
  output; a zero router weight contributes nothing; E = k = 1 gives shared + FFN.
* Backward: central finite differences in float64 for every gradient the layer returns.
"""

import math

import numpy as np
import pytest

import oracle


def test_silu_closed_form_points():
    ln3 = math.log(3.0)
    z = np.array([0.0, ln3, -ln3, 60.0, -60.0])
    s = oracle.silu(z)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(0.75 * ln3, rel=1e-15)      # sigmoid(ln 3) = 3/4
    assert s[2] == pytest.approx(-0.25 * ln3, rel=1e-15)     # sigmoid(-ln 3) = 1/4
    assert s[3] == pytest.approx(60.0, rel=1e-15)
    assert abs(s[4]) < 1e-20


def _perm_matrix(perm, scale=1.0):
    n = len(perm)
    P = np.zeros((n, n))
    for i, p in enumerate(perm):
        P[i, p] = scale        # x @ P moves x[i] to column p
    return P


def test_expert_ffn_with_permutation_weights():
    n = 5
    x = np.array([[0.5, -1.25, 2.0, 0.0, 3.5], [1.0, 2.0, -0.5, 0.75, -2.0]])
    pg, pu, pd = [2, 0, 4, 1, 3], [1, 3, 0, 4, 2], [4, 2, 3, 0, 1]
    a = 0.7
    Wg, Wu, Wd = _perm_matrix(pg, a), _perm_matrix(pu), _perm_matrix(pd)
    g, u, h, y = oracle.expert_ffn(x, Wg, Wu, Wd)
    for r in range(2):
        gv, uv = np.zeros(n), np.zeros(n)
        for i in range(n):
            gv[pg[i]] = a * x[r, i]
            uv[pu[i]] = x[r, i]
        hv = [gv[f] / (1.0 + math.exp(-gv[f])) * uv[f] for f in range(n)]
        yv = np.zeros(n)
        for f in range(n):
            yv[pd[f]] = hv[f]
        np.testing.assert_allclose(g[r], gv, rtol=0, atol=0)
        np.testing.assert_allclose(u[r], uv, rtol=0, atol=0)
        np.testing.assert_allclose(y[r], yv, rtol=1e-15, atol=1e-15)


def test_expert_ffn_zero_gate_and_linearity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4, 6))
    Wg, Wu, Wd = rng.standard_normal((6, 3)), rng.standard_normal((6, 3)), rng.standard_normal((3, 6))
    assert (oracle.expert_ffn(x, np.zeros_like(Wg), Wu, Wd)[3] == 0).all()
    y = oracle.expert_ffn(x, Wg, Wu, Wd)[3]
    np.testing.assert_allclose(oracle.expert_ffn(x, Wg, 2 * Wu, Wd)[3], 2 * y, rtol=1e-14)
    np.testing.assert_allclose(oracle.expert_ffn(x, Wg, Wu, -3 * Wd)[3], -3 * y, rtol=1e-14)


def _layer(T=12, d=8, E=4, k=2, F=6, Fs=5, seed=0, shared=True):
    rng = np.random.default_rng(seed)
    L = dict(
        x=rng.standard_normal((T, d)),
        Wr=rng.standard_normal((d, E)) * 0.7,
        b=rng.standard_normal(E) * 0.1,
        Wg=rng.standard_normal((E, d, F)) * 0.4,
        Wu=rng.standard_normal((E, d, F)) * 0.4,
        Wd=rng.standard_normal((E, F, d)) * 0.4,
        shared=(rng.standard_normal((d, Fs)) * 0.4, rng.standard_normal((d, Fs)) * 0.4,
                rng.standard_normal((Fs, d)) * 0.4) if shared else None,
        dY=rng.standard_normal((T, d)),
        k=k,
    )
    return L


def test_identical_experts_with_k_equal_E_reduce_to_one_ffn():
    L = _layer(E=4, k=4)
    Wg = np.repeat(L["Wg"][:1], 4, axis=0)
    Wu = np.repeat(L["Wu"][:1], 4, axis=0)
    Wd = np.repeat(L["Wd"][:1], 4, axis=0)
    _, _, idx, w = oracle.route(L["x"], L["Wr"], L["b"], 4)
    y = oracle.moe_forward(L["x"], Wg, Wu, Wd, L["shared"], idx, w)
    want = oracle.expert_ffn(L["x"], *L["shared"])[3] + oracle.expert_ffn(L["x"], Wg[0], Wu[0], Wd[0])[3]
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_single_expert_layer():
    L = _layer(E=1, k=1)
    _, _, idx, w = oracle.route(L["x"], L["Wr"], L["b"], 1)
    assert (w == 1.0).all()
    y = oracle.moe_forward(L["x"], L["Wg"], L["Wu"], L["Wd"], L["shared"], idx, w)
    want = oracle.expert_ffn(L["x"], *L["shared"])[3] + oracle.expert_ffn(L["x"], L["Wg"][0], L["Wu"][0], L["Wd"][0])[3]
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


def test_token_permutation_permutes_output():
    L = _layer(T=10)
    _, _, idx, w = oracle.route(L["x"], L["Wr"], L["b"], L["k"])
    y = oracle.moe_forward(L["x"], L["Wg"], L["Wu"], L["Wd"], L["shared"], idx, w)
    perm = np.random.default_rng(1).permutation(10)
    _, _, idx_p, w_p = oracle.route(L["x"][perm], L["Wr"], L["b"], L["k"])
    y_p = oracle.moe_forward(L["x"][perm], L["Wg"], L["Wu"], L["Wd"], L["shared"], idx_p, w_p)
    np.testing.assert_allclose(y_p, y[perm], rtol=1e-13, atol=1e-13)


def test_zero_router_weight_contributes_nothing():
    L = _layer()
    _, _, idx, w = oracle.route(L["x"], L["Wr"], L["b"], 2)
    w0 = w.copy()
    w0[:, 1] = 0.0
    y = oracle.moe_forward(L["x"], L["Wg"], L["Wu"], L["Wd"], L["shared"], idx, w0)
    y1 = oracle.moe_forward(L["x"], L["Wg"], L["Wu"], L["Wd"], L["shared"], idx[:, :1], w0[:, :1])
    np.testing.assert_allclose(y, y1, rtol=1e-14, atol=1e-14)
    # no shared expert and all weights zero: the output is exactly zero
    yz = oracle.moe_forward(L["x"], L["Wg"], L["Wu"], L["Wd"], None, idx, np.zeros_like(w))
    assert (yz == 0).all()


# ------------------------------- backward: finite differences -------------------------------

def _loss(L, x, Wr, b, Wg, Wu, Wd, shared, idx):
    logits = oracle.router_logits(x, Wr, b)
    y = oracle.moe_forward_from_logits(x, logits, idx, Wg, Wu, Wd, shared)
    return float((y * L["dY"]).sum())


def _fd(f, arr, h=1e-6):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + h
        fp = f()
        arr[i] = old - h
        fm = f()
        arr[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("shared", [True, False])
def test_backward_matches_finite_differences(shared):
    L = _layer(T=6, d=5, E=4, k=2, F=3, Fs=4, seed=7, shared=shared)
    logits = oracle.router_logits(L["x"], L["Wr"], L["b"])
    idx = oracle.topk_select(logits.astype(np.float32), L["k"])
    assert oracle.topk_gap(logits.astype(np.float32), L["k"]).min() > 1e-3, "no near ties"
    sh = [a.copy() for a in L["shared"]] if shared else None
    x, Wr, b = L["x"].copy(), L["Wr"].copy(), L["b"].copy()
    Wg, Wu, Wd = L["Wg"].copy(), L["Wu"].copy(), L["Wd"].copy()

    def f():
        return _loss(L, x, Wr, b, Wg, Wu, Wd, sh, idx)

    got = oracle.moe_backward(x, L["dY"], Wr, Wg, Wu, Wd, sh, logits, idx)
    tol = dict(rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(got["dX"], _fd(f, x), **tol)
    np.testing.assert_allclose(got["dW_router"], _fd(f, Wr), **tol)
    np.testing.assert_allclose(got["dW_gate"], _fd(f, Wg), **tol)
    np.testing.assert_allclose(got["dW_up"], _fd(f, Wu), **tol)
    np.testing.assert_allclose(got["dW_down"], _fd(f, Wd), **tol)
    if shared:
        np.testing.assert_allclose(got["dWs_gate"], _fd(f, sh[0]), **tol)
        np.testing.assert_allclose(got["dWs_up"], _fd(f, sh[1]), **tol)
        np.testing.assert_allclose(got["dWs_down"], _fd(f, sh[2]), **tol)
    # gradient with respect to the router logits themselves (selection held constant)
    lg = logits.copy()

    def fl():
        y = oracle.moe_forward_from_logits(x, lg, idx, Wg, Wu, Wd, sh)
        return float((y * L["dY"]).sum())

    dl_fd = _fd(fl, lg)
    np.testing.assert_allclose(got["dlogits"], dl_fd, **tol)
    # unselected experts get exactly zero; the bias gradient is the column sum of dlogits
    mask = np.ones_like(logits, dtype=bool)
    np.put_along_axis(mask, idx.astype(np.int64), False, axis=1)
    assert (got["dlogits"][mask] == 0).all()
    np.testing.assert_allclose(got["dlogits"].sum(axis=0), _fd(f, b), **tol)
