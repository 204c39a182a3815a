"""Pins of the oracle's NVFP4 quantiser and forward reading (CPU).

Quantiser (oracle/nvfp4.py): E2M1 elements, one E4M3 scale per 16 along the reduction
dimension, one fp32 tensor scale (the format NVIDIA defines as NVFP4; the first page names it as
the format of the authors' earlier kernels).
* Exhaustive: the 16 codes and their values.
* Brute force: E2M1 rounding equals a nearest search over the eight magnitudes with ties to the
  even code, on random values and every midpoint; saturation at 6.
* Closed forms: the tensor scale S = 2688 / A (S = 1 for A = 0); blocks of values q * s * g
  are fixed points; values above a calibrated amax clip to it; power-of-two scaling of a tensor
  leaves its codes unchanged.
* Axes: an outlier coarsens only its own block of 16 along the last axis.

Forward (oracle.moe_forward_nvfp4): which outputs an outlier planted in x, in a weight, or in
h changes shows the axis every operand is quantised along (fixture below); zero down weights
give zero; the distance to the float64 forward on random data.
"""

import numpy as np

import oracle
from oracle.moe import _nv_weight


# ------------------------------------------------------------------ quantiser

def test_codes():
    vals = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert vals[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert (vals[8:] == -vals[:8]).all() and np.signbit(vals[8])
    back = oracle.e2m1_encode(vals)
    assert back[:8].tolist() == list(range(8))
    assert back[9:].tolist() == list(range(9, 16))
    assert back[8] == 0          # -0 has no negative product: the sign bit is v < 0


def _brute(v):
    """Nearest of the eight magnitudes, ties to the even index, saturating; sign v < 0."""
    a = np.abs(v)
    d = np.abs(a[:, None] - oracle.E2M1_VALUES[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    idx = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    idx = np.where(a > 6.0, 7, idx)
    return (idx | np.where(v < 0, 8, 0)).astype(np.uint8)


def test_e2m1_rounding_brute_force():
    rng = np.random.default_rng(0)
    g = oracle.E2M1_VALUES
    mids = (g[:-1] + g[1:]) / 2
    v = np.concatenate([rng.uniform(-8, 8, 50000), mids, -mids, g, -g[1:],
                        np.nextafter(mids, 0), np.nextafter(mids, 10), [6.5, 7.0, 100.0, -1e9]])
    v = v.astype(np.float32).astype(np.float64)
    assert (oracle.e2m1_encode(v) == _brute(v)).all()
    # the ties, one by one (ties go to 0, 1, 1, 2, 2, 4, 4)
    ties = oracle.e2m1_encode(mids)
    assert oracle.e2m1_decode(ties).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_tensor_scale():
    S, g = oracle.nv_tensor_scale(2688.0)
    assert S == 1.0 and g == 1.0
    S, g = oracle.nv_tensor_scale(0.0)
    assert S == 1.0 and g == 1.0
    S, g = oracle.nv_tensor_scale(3.0)
    assert S == np.float32(896.0) and g == np.float32(1.0) / np.float32(896.0)
    S, g = oracle.nv_tensor_scale(7.0)          # 384 = 2688 / 7 exactly
    assert S == np.float32(384.0)


def _fixed_point_tensor(rng, rows, K, A_exp):
    """Blocks of q * s * g with the tensor amax 2688 * 2^A_exp: each block holds a +-6 code,
    so its amax is 6 s and (a / 6) S = s exactly."""
    nb = K // 16
    sc = rng.integers(0x20, 0x7F, size=(rows, nb)).astype(np.uint8)      # E4M3 scales 2^-3 .. 448
    sc[0, 0] = 0x7E                                                      # one block at 448
    q = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    q[:, ::16] = np.where(rng.random((rows, nb)) < 0.5, 7, 15)           # a +-6 in every block
    g = np.float32(2.0 ** A_exp)
    v = oracle.e2m1_decode(q) * np.repeat(oracle.e4m3_decode(sc), 16, axis=1) * np.float64(g)
    return v, q, sc, g


def test_fixed_points():
    rng = np.random.default_rng(1)
    for A_exp in (0, -7, 5):
        v, q, sc, g = _fixed_point_tensor(rng, 6, 128, A_exp)
        q2, sc2, g2 = oracle.nv_quantize(v)
        assert g2 == g
        assert (sc2 == sc).all()
        # codes agree except that -0 encodes as +0
        assert ((q2 == q) | ((q == 8) & (q2 == 0))).all()
        assert (oracle.nv_dequantize(q2, sc2, g2) == v).all()


def test_power_of_two_scaling_keeps_the_codes():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((5, 64)) * rng.uniform(0.01, 3, (5, 1))).astype(np.float32).astype(np.float64)
    q0, s0, g0 = oracle.nv_quantize(v)
    for k in (-9, -1, 3, 11):
        q1, s1, g1 = oracle.nv_quantize(v * 2.0 ** k)
        assert (q1 == q0).all() and (s1 == s0).all() and g1 == np.float32(g0 * 2.0 ** k)


def test_block_axis_and_error_bound():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((4, 64)).astype(np.float32).astype(np.float64)
    v[3, 5] = 0.0
    anchor = 64.0 * np.abs(v).max()
    v[0, 63] = anchor                                  # keeps the tensor amax below fixed
    q0, s0, g0 = oracle.nv_quantize(v)
    d0 = oracle.nv_dequantize(q0, s0, g0)
    # error bound: at most half a step of the block's grid (step <= 2 s_val g)
    sv = np.repeat(oracle.e4m3_decode(s0), 16, axis=1) * np.float64(g0)
    assert (np.abs(d0 - v) <= sv + 1e-12).all()
    # an outlier in row 1, column 20 (block 1) coarsens row 1's block 1 only
    w = v.copy()
    w[1, 20] = 16.0 * np.abs(v[:, :63]).max()
    q1, s1, g1 = oracle.nv_quantize(w)
    assert g1 == g0
    d1 = oracle.nv_dequantize(q1, s1, g1)
    changed = np.abs(d1 - d0) > 0
    changed[1, 20] = False
    assert changed[1, 16:32].any()
    keep = np.ones_like(changed)
    keep[1, 16:32] = False
    assert not changed[keep].any()


def test_calibrated_amax_clips():
    v = np.zeros((1, 32))
    v[0, 0], v[0, 1], v[0, 16] = 40.0, -3.0, 0.5
    q, sc, g = oracle.nv_quantize(v, tensor_amax=10.0)
    d = oracle.nv_dequantize(q, sc, g)
    assert d[0, 0] == np.float64(np.float32(448.0 * 6.0) * np.float64(g))   # the largest value
    assert abs(d[0, 0] - 10.0) < 1e-5
    assert sc[0, 0] == 0x7E                                                  # scale saturated
    assert abs(d[0, 16] - 0.5) <= 0.25 * 0.5                                # other block intact


def test_zero_tensor():
    q, sc, g = oracle.nv_quantize(np.zeros((2, 32)))
    assert (q == 0).all() and (sc == 0).all() and g == 1.0


def test_weight_quantiser_runs_along_k():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((64, 48)) * 0.5
    W[63, 47] = 40.0                                   # anchor: the tensor amax
    base = _nv_weight(W)
    W2 = W.copy()
    W2[21, 5] = 8.0                                    # K block 1 (rows 16..31) of column 5
    moved = np.abs(_nv_weight(W2) - base) > 0
    moved[21, 5] = False
    assert moved[16:32, 5].any()
    keep = np.ones_like(moved)
    keep[16:32, 5] = False
    assert not moved[keep].any()


# ------------------------------------------------------------------ forward axes
# Fixture: 8 tokens; token t has a one-hot value a_t at column 16 t of x (its own 16-block of
# d), and every token has small values at columns 35 and 36 (block 2 of its row).  Anchors fix
# the tensor amax of x (x[7, 120] = 64, the calibrated amax_x too) and of every weight (32 at a
# corner no plant touches), so a plant moves no tensor scale.  One expert, k = 1, no shared
# expert; h takes a calibrated amax_h.

T, D, F = 8, 128, 32
AMAX_X, AMAX_H = 64.0, 6.0
IDX = np.zeros((T, 1), dtype=np.int32)
W1 = np.ones((T, 1))


def _fixture(seed=5):
    rng = np.random.default_rng(seed)
    x = np.zeros((T, D))
    x[np.arange(T), 16 * np.arange(T)] = rng.uniform(0.7, 1.6, size=T)
    x[:, 35] = rng.uniform(0.05, 0.1, size=T)
    x[:, 36] = rng.uniform(0.05, 0.1, size=T)
    x[7, 120] = AMAX_X
    Wg = rng.standard_normal((D, F)) * 0.5
    Wu = rng.standard_normal((D, F)) * 0.5
    Wd = rng.standard_normal((F, D)) * 0.2
    Wg[127, 31] = Wu[127, 31] = 32.0
    Wd[31, 127] = 32.0
    return x, Wg, Wu, Wd


def _fwd(x, Wg, Wu, Wd):
    return oracle.moe_forward_nvfp4(x, Wg[None], Wu[None], Wd[None], None, IDX, W1, AMAX_X, AMAX_H)


def _rows_moved(a, b):
    return [t for t in range(T) if not np.array_equal(a[t], b[t])]


def test_forward_x_along_d():
    # the plant at column 36 multiplies zero weight rows, so only the coarsening of its block's
    # other values (token 2's one-hot value at column 32 and column 35) can reach y
    x, Wg, Wu, Wd = _fixture()
    Wg[36, :] = 0.0
    Wu[36, :] = 0.0
    base = _fwd(x, Wg, Wu, Wd)
    x2 = x.copy()
    x2[2, 36] = 16.0            # block 2 of token 2's row
    assert _rows_moved(_fwd(x2, Wg, Wu, Wd), base) == [2]


def test_forward_gate_and_up_weights_along_d():
    x, Wg, Wu, Wd = _fixture()
    base = _fwd(x, Wg, Wu, Wd)
    for which in (0, 1):
        W = [Wg.copy(), Wu.copy()]
        W[which][53, 20] = 8.0  # K block 3 (rows 48..63): row 48 is token 3's, row 53 nobody's
        assert _rows_moved(_fwd(x, W[0], W[1], Wd), base) == [3]


def test_forward_down_weight_along_F():
    x, Wg, Wu, Wd = _fixture()
    base = _fwd(x, Wg, Wu, Wd)
    Wd2 = Wd.copy()
    Wd2[5, 60] = 8.0            # F block 0 of column 60
    y = _fwd(x, Wg, Wu, Wd2)
    cols = [j for j in range(D) if not np.array_equal(y[:, j], base[:, j])]
    assert cols == [60]


def test_forward_h_along_F():
    # a large u[3, 3] (through token 3's row 48 of W_up) makes h[3, 3] an outlier of F block 0
    # of token 3's h row; W_down row 3 is zero, so only the coarsening of the block's other
    # values can reach y
    x, Wg, Wu, Wd = _fixture()
    Wd[3, :] = 0.0
    base = _fwd(x, Wg, Wu, Wd)
    Wu2 = Wu.copy()
    Wu2[48, 3] = 8.0
    assert _rows_moved(_fwd(x, Wg, Wu2, Wd), base) == [3]


def test_forward_zero_down_weights():
    x, Wg, Wu, Wd = _fixture()
    assert (_fwd(x, Wg, Wu, np.zeros_like(Wd)) == 0).all()


def test_forward_close_to_float64():
    rng = np.random.default_rng(6)
    Tn, d, E, k, Fn = 48, 256, 4, 2, 128
    x = rng.standard_normal((Tn, d)).astype(np.float32).astype(np.float64)
    Wg = rng.standard_normal((E, d, Fn)) / np.sqrt(d)
    Wu = rng.standard_normal((E, d, Fn)) / np.sqrt(d)
    Wd = rng.standard_normal((E, Fn, d)) / np.sqrt(Fn)
    sh = (rng.standard_normal((d, Fn)) / np.sqrt(d), rng.standard_normal((d, Fn)) / np.sqrt(d),
          rng.standard_normal((Fn, d)) / np.sqrt(Fn))
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(Tn)]).astype(np.int32)
    w = rng.uniform(0.2, 0.8, (Tn, k))
    ref = oracle.moe_forward(x, Wg, Wu, Wd, sh, idx, w)
    amax_h = 4.0
    got = oracle.moe_forward_nvfp4(x, Wg, Wu, Wd, sh, idx, w, np.abs(x).max(), amax_h)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    # four quantised operands of about 3 significant bits each: a few per cent, never exact
    assert 0.01 < rel < 0.25, rel
