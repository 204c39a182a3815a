"""Shared helpers of the test suite (comparison metrics, library loading, input plumbing)."""

import os

import numpy as np
import torch

import mixture_experts_layer_14_gb300 as mok

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances for bf16 outputs and gradients against the float64 oracle.
MAX_REL = 2e-2      # max|gpu - ref| <= MAX_REL * max|ref|
MEAN_REL = 5e-3     # sum|gpu - ref| / sum|ref| <= MEAN_REL
NEAR_TIE = 1e-4     # tokens whose k-th / (k+1)-th float32 logit gap is below this are excluded


def ensure_lib():
    if not os.path.exists(mok.lib_path()):
        from mixture_experts_layer_14_gb300 import build

        build.build()
    return mok.lib()


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    scale = np.abs(ref).max()
    max_rel = d.max() / scale if scale > 0 else d.max()
    mean_rel = d.sum() / np.abs(ref).sum() if np.abs(ref).sum() > 0 else d.sum()
    return float(max_rel), float(mean_rel)


def assert_close(name, got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL):
    mx, mn = errors(got, ref)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{name}: non-finite values"
    assert mx <= max_rel and mn <= mean_rel, f"{name}: max_rel={mx:.3e} mean_rel={mn:.3e}"
    return mx, mn


def to_dev(layer, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in layer.items()}


def dims_of(shape, T=None, dtype=mok.MOK_BF16):
    return mok.dims(shape.T if T is None else T, shape.d, shape.E, shape.k, shape.F,
                    shape.F_shared, shape.n_shared, dtype)


class LazyExperts:
    """Indexable view of a stacked [E, a, b] bf16 tensor that converts one expert to float64 on
    access (the oracle's weights on large layers)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return f64(self.t[e])
