"""Pins of the oracle's MXFP8 quantiser (E4M3 values, UE8M0 scale per 32 elements), on the CPU.

* Exhaustive: every E4M3 code decodes to a value that encodes back to the same code.
* Library special case: encoding agrees bit for bit with the torch.float8_e4m3fn conversion
  routine on random and edge values inside the finite range.
* Closed forms: saturation to +-448, the scale of blocks whose amax is 448 * 2^s exactly or just
  above it, the all-zero block, and the half-ulp bound of quantise -> dequantise.
"""

import numpy as np
import pytest
import torch

import oracle


def test_all_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    nan = np.isnan(vals)
    assert sorted(codes[nan].tolist()) == [0x7F, 0xFF]
    back = oracle.e4m3_encode(vals)
    assert (back[~nan] == codes[~nan]).all()
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    # known values of the format: 1.0 = 0x38, -2.0 = 0xC0, 0.5 = 0x30
    assert oracle.e4m3_encode(np.array([1.0, -2.0, 0.5])).tolist() == [0x38, 0xC0, 0x30]


def _torch_e4m3(v32):
    return torch.from_numpy(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_library_conversion():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)
    ]
    # exact midpoints between neighbouring codes exercise ties-to-even
    pos = oracle.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    parts += [mids, -mids, pos.astype(np.float32), np.array([0.0, -0.0, 448.0, -448.0], np.float32)]
    v = np.concatenate(parts)
    v = v[np.abs(v) <= 448.0]
    got = oracle.e4m3_encode(v.astype(np.float64))
    want = _torch_e4m3(v)
    assert (got == want).all(), np.nonzero(got != want)[0][:10]


def test_saturation():
    got = oracle.e4m3_encode(np.array([449.0, 1e6, -500.0, np.inf, -np.inf]))
    assert got.tolist() == [0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_scale_rule_closed_forms():
    s = np.array([-10, -1, 0, 3, 20])
    exact = 448.0 * np.exp2(s)
    assert (oracle.mx_scale_exponent(exact) == s).all()
    above = np.nextafter(exact.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    assert (oracle.mx_scale_exponent(above) == s + 1).all()
    assert oracle.mx_scale_exponent(np.array([0.0]))[0] == -127
    assert oracle.mx_scale_exponent(np.array([1e-300]))[0] == -127     # clamped
    # amax = 1 -> 448 * 2^-8 = 1.75 >= 1 > 0.875: s = -8
    assert oracle.mx_scale_exponent(np.array([1.0]))[0] == -8


def test_quantize_block_layout_and_error_bound():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal((3, 96)) * np.array([[1e-4], [1.0], [1e3]])).astype(np.float32).astype(np.float64)
    v[1, 32:64] = 0.0
    q, sb = oracle.mx_quantize(v)
    assert q.shape == (3, 96) and sb.shape == (3, 3)
    assert sb[1, 1] == 0 and (q[1, 32:64] == 0).all()
    deq = oracle.mx_dequantize(q, sb)
    for r in range(3):
        for b in range(3):
            blk = v[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            if amax == 0:
                continue
            s = int(sb[r, b]) - 127
            assert 448.0 * 2.0 ** (s - 1) < amax <= 448.0 * 2.0 ** s
            # nearest rounding: error at most half the spacing at each magnitude (3 mantissa bits)
            err = np.abs(deq[r, 32 * b:32 * b + 32] - blk)
            spacing = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(blk) / 2.0 ** s, 2.0 ** -6))) - 3), 2.0 ** -9)
            assert (err <= 0.5 * spacing * 2.0 ** s * (1 + 1e-12)).all()


def _representable(rng, shape):
    """Values exactly representable in MXFP8 blocks: small integers times a power of two."""
    return rng.integers(-7, 8, size=shape).astype(np.float64) * 2.0 ** rng.integers(-3, 1)


def test_mxfp8_forward_pins():
    rng = np.random.default_rng(3)
    T, d, E, k, F = 6, 64, 3, 2, 32
    x = _representable(rng, (T, d))
    Wg = np.stack([_representable(rng, (d, F)) * 0.125 for _ in range(E)])
    Wu = np.stack([_representable(rng, (d, F)) * 0.125 for _ in range(E)])
    Wd = np.zeros((E, F, d))
    idx = np.array([[0, 1], [1, 2], [2, 0], [0, 2], [1, 0], [2, 1]], dtype=np.int32)
    w = rng.random((T, k))
    # representable inputs are not changed by the quantiser, so with a zero W_down only the
    # shared expert remains; its gate/up products equal the float64 ones
    sh = (_representable(rng, (d, F)) * 0.125, _representable(rng, (d, F)) * 0.125, np.zeros((F, d)))
    assert (oracle.moe_forward_mxfp8(x, Wg, Wu, Wd, sh, idx, w) == 0).all()
    assert (oracle.mx_dequantize(*oracle.mx_quantize(x)) == x).all()
    # with random data the MXFP8 output stays within a few E4M3 steps of the float64 output
    x = rng.standard_normal((T, d))
    Wg, Wu = rng.standard_normal((E, d, F)) / 8, rng.standard_normal((E, d, F)) / 8
    Wd = rng.standard_normal((E, F, d)) / 6
    sh = (rng.standard_normal((d, F)) / 8, rng.standard_normal((d, F)) / 8, rng.standard_normal((F, d)) / 6)
    y = oracle.moe_forward(x, Wg, Wu, Wd, sh, idx, w)
    yq = oracle.moe_forward_mxfp8(x, Wg, Wu, Wd, sh, idx, w)
    rel = np.abs(yq - y).max() / np.abs(y).max()
    assert 1e-4 < rel < 0.1


def test_token_axis_quantiser_matches_columnwise_quantiser():
    """The weight-gradient operands are quantised along tokens: each column of A[n, C] in blocks
    of 32 rows from row 0, the last block zero-padded.  Checked column by column against the
    pinned quantiser on a padded vector."""
    from oracle.moe import _mx_qd_tokens

    rng = np.random.default_rng(4)
    A = rng.standard_normal((70, 5)) * np.exp2(rng.integers(-8, 8, size=(70, 1)))
    got = _mx_qd_tokens(A)
    for j in range(A.shape[1]):
        col = np.concatenate([A[:, j], np.zeros(26)])
        want = oracle.mx_dequantize(*oracle.mx_quantize(col[None, :]))[0, :70]
        assert (got[:, j] == want).all()
    # a large token in block 0 coarsens its block's other values but not block 1's
    B = A.copy()
    B[3, :] *= 2.0 ** 12
    q = _mx_qd_tokens(B)
    assert (q[32:64] == got[32:64]).all()
    assert (q[[0, 1, 2, 4]] != got[[0, 1, 2, 4]]).any()


def _small_backward_case(rng, representable):
    T, d, E, k, F = 40, 64, 3, 2, 64
    if representable:
        x = _representable(rng, (T, d))
        dY = _representable(rng, (T, d))
        Wg = np.stack([_representable(rng, (d, F)) / 16 for _ in range(E)])
        Wu = np.stack([_representable(rng, (d, F)) / 16 for _ in range(E)])
        Wd = np.stack([_representable(rng, (F, d)) / 16 for _ in range(E)])
        sh = tuple(_representable(rng, s) / 16 for s in ((d, F), (d, F), (F, d)))
        Wr = _representable(rng, (d, E)) / 16
    else:
        x = rng.standard_normal((T, d))
        dY = rng.standard_normal((T, d))
        Wg, Wu = rng.standard_normal((E, d, F)) / 8, rng.standard_normal((E, d, F)) / 8
        Wd = rng.standard_normal((E, F, d)) / 8
        sh = (rng.standard_normal((d, F)) / 8, rng.standard_normal((d, F)) / 8,
              rng.standard_normal((F, d)) / 8)
        Wr = rng.standard_normal((d, E)) / 8
    logits = x @ Wr
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    return x, dY, Wr, Wg, Wu, Wd, sh, logits, idx


def test_mxfp8_backward_within_e4m3_steps_of_float64():
    """Every gradient of the MXFP8 reading is within a few E4M3 steps of the float64 backward
    (pinned by finite differences) and not equal to it: a dropped or transposed term would be an
    O(1) error, a missing quantisation point an exact match."""
    rng = np.random.default_rng(5)
    args = _small_backward_case(rng, representable=False)
    ref = oracle.moe_backward(*args)
    got = oracle.moe_backward_mxfp8(*args)
    for key in ("dX", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down",
                "dlogits", "dW_router"):
        rel = np.abs(got[key] - ref[key]).max() / np.abs(ref[key]).max()
        assert 1e-4 < rel < 0.15, (key, rel)


def test_mxfp8_backward_router_path_exact_on_representable_inputs():
    """With x, dY and every weight exactly representable in MXFP8, q_d(dY) q_d(W_down)^T and the
    forward's gate/up products are the float64 ones, so the router-weight gradients <a, h>,
    dlogits and dW_router equal the float64 backward's; the weight gradients do not (dG, dU and
    w h are quantised)."""
    rng = np.random.default_rng(6)
    args = _small_backward_case(rng, representable=True)
    ref = oracle.moe_backward(*args)
    got = oracle.moe_backward_mxfp8(*args)
    for key in ("dw", "dlogits", "dW_router"):
        assert np.allclose(got[key], ref[key], rtol=1e-12, atol=1e-12 * np.abs(ref[key]).max()), key
    assert not np.allclose(got["dW_gate"], ref["dW_gate"], rtol=1e-6, atol=0)
    zero = oracle.moe_backward_mxfp8(args[0], np.zeros_like(args[1]), *args[2:])
    for key in ("dX", "dW_gate", "dW_up", "dW_down", "dlogits"):
        assert not zero[key].any(), key
