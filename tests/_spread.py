"""Power-of-two magnitude spread for MXFP8 parity inputs (test infrastructure).

MXFP8 keeps one scale per 32 elements along a GEMM's reduction dimension, and a value's rounding
depends on its block only when the block mixes magnitudes more than about 2^15 apart.  This
rescales a layer by exact powers of two so that every quantised operand mixes such magnitudes
along its reduction dimension while the float64 layer stays the same function:

    x[:, i] * 2^r[i]          W_router[i, :], W_gate[e, i, :] * 2^-r[i]
    W_up[e, i, f] * 2^(c[e, f] - r[i])     W_down[e, f, j] * 2^-(c[e, f] + q[j])
    dY[:, j] * 2^q[j]         (the shared expert likewise with its own c)

g, u / 2^c, h / 2^c and the logits are then unchanged, and every output or gradient is the
unspread one times a known power of two per row or column, so both sides of a comparison can be
unscaled exactly before the usual bars apply.  An operand quantised along the wrong axis would
see no spread inside its blocks (each factor is constant along the other axis) and would round
differently at O(1).
"""

import numpy as np
import torch


def spread_factors(shape, R, seed):
    rng = np.random.default_rng(seed)
    E, d, F, Fs = shape.E, shape.d, shape.F, shape.F_shared
    return {"r": rng.integers(-R, R + 1, size=d), "c": rng.integers(-R, R + 1, size=(E, F)),
            "cs": rng.integers(-R, R + 1, size=max(Fs, 1)),
            "q": rng.integers(-R, R + 1, size=d) if shape.backward else np.zeros(d, dtype=np.int64)}


def _scaled(t, e):
    """t (bf16) times 2^e elementwise, exact (e broadcast to t's shape)."""
    return (t.to(torch.float64) * torch.from_numpy(np.exp2(e.astype(np.float64)))).to(torch.bfloat16)


def apply_spread(L, s):
    """A copy of the CPU layer dict L rescaled by the factors s (see the module docstring)."""
    r, c, cs, q = s["r"], s["c"], s["cs"], s["q"]
    out = dict(L)
    out["x"] = _scaled(L["x"], r[None, :])
    out["W_router"] = _scaled(L["W_router"], -r[:, None])
    out["W_gate"] = _scaled(L["W_gate"], -r[None, :, None])
    out["W_up"] = _scaled(L["W_up"], c[:, None, :] - r[None, :, None])
    out["W_down"] = _scaled(L["W_down"], -(c[:, :, None] + q[None, None, :]))
    if L.get("Ws_gate") is not None:
        Fs = L["Ws_gate"].shape[1]
        out["Ws_gate"] = _scaled(L["Ws_gate"], -r[:, None])
        out["Ws_up"] = _scaled(L["Ws_up"], cs[None, :Fs] - r[:, None])
        out["Ws_down"] = _scaled(L["Ws_down"], -(cs[:Fs, None] + q[None, :]))
    if L.get("dY") is not None:
        out["dY"] = _scaled(L["dY"], q[None, :])
    return out


def unscale(key, a, s):
    """Output or gradient `key` of the spread layer mapped back to the unspread layer's scale."""
    r, c, cs, q = s["r"], s["c"], s["cs"], s["q"]
    a = np.asarray(a, dtype=np.float64)
    if key == "y":
        return a * np.exp2(q)[None, :]
    if key == "dX":
        return a * np.exp2(r)[None, :]
    if key == "dW_gate":
        return a * np.exp2(-r)[None, :, None]
    if key == "dW_up":
        return a * np.exp2(c[:, None, :] - r[None, :, None])
    if key == "dW_down":
        return a * np.exp2(-(c[:, :, None] + q[None, None, :]))
    Fs = a.shape[1] if key in ("dWs_gate", "dWs_up") else a.shape[0]
    if key == "dWs_gate":
        return a * np.exp2(-r)[:, None]
    if key == "dWs_up":
        return a * np.exp2(cs[None, :Fs] - r[:, None])
    if key == "dWs_down":
        return a * np.exp2(-(cs[:Fs, None] + q[None, :]))
    if key == "dW_router":
        return a * np.exp2(-r)[:, None]
    if key in ("dlogits", "dw"):
        return a
    raise KeyError(key)
