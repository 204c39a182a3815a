"""Seeded synthetic inputs for the MoE layer (shared by the tests, the oracle checks and the bench).

This module holds no arithmetic of the method: it only draws seeded random tensors with the
shapes and distributions of the layer workloads and rounds them to bf16.  Every tensor has its
own seed (x: 1000+c, W_router: 2000+c, W_gate: 3000+c, W_up: 4000+c, W_down: 5000+c, shared
expert: 6000+c, bias: 7000+c, expert-rank permutation: 8000+c, dY: 9000+c, c = workload number).

Layouts: x[T,d], W_router[d,E], W_gate/W_up[E,d,F], W_down[E,F,d], Ws_gate/Ws_up[d,Fs],
Ws_down[Fs,d], bias[E] float32 or None, dY[T,d].
"""

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    F_shared: int
    n_shared: int = 1
    weight_std: float = 0.0      # 0 -> N(0, 1/sqrt(fan_in))
    bias: str = "none"           # "none" | "normal0.1" | "zipf"
    dtype: str = "bf16"          # arithmetic of the expert GEMMs: "bf16" | "mxfp8" | "nvfp4"
    backward: bool = False
    cid: int = 0                 # seed offset

    @property
    def R(self):
        return self.T * self.k

    def with_(self, **kw):
        return replace(self, **kw)


# The layer workloads (sizes of DeepSeek-V3 / Kimi-class MoE layers, plus a tiny one).
WORKLOADS = {
    "tiny": LayerShape("tiny", 256, 256, 8, 2, 128, 128, 1, 0.02, "none", "bf16", False, 1),
    "dsv3_bf16_fwd": LayerShape("dsv3_bf16_fwd", 4096, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                "normal0.1", "bf16", False, 2),
    "kimi_skew_bf16_fwd": LayerShape("kimi_skew_bf16_fwd", 16384, 7168, 384, 8, 2048, 2048, 1,
                                     0.0, "zipf", "bf16", False, 3),
    "dsv3_mxfp8_fwd": LayerShape("dsv3_mxfp8_fwd", 8192, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                 "normal0.1", "mxfp8", False, 4),
    "dsv3_bf16_train": LayerShape("dsv3_bf16_train", 8192, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                  "normal0.1", "bf16", True, 5),
    # the training step with every expert GEMM block-scaled (forward and backward)
    "dsv3_mxfp8_train": LayerShape("dsv3_mxfp8_train", 8192, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                   "normal0.1", "mxfp8", True, 10),
    # decode-sized batch of the same layer: 64 tokens (512 routes) still touch most experts, so
    # the step streams nearly all the expert weights for few rows each
    "dsv3_decode_t64": LayerShape("dsv3_decode_t64", 64, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                  "normal0.1", "bf16", False, 9),
    # A slice of the DeepSeek-V3 layer with the same rows per expert (T*k/E = 128) but 32
    # experts, so that a full profiler capture holds a few GB on the device.
    "dsv3_slice_e32": LayerShape("dsv3_slice_e32", 512, 7168, 32, 8, 2048, 2048, 1, 0.0,
                                 "normal0.1", "bf16", False, 6),
    # the same kind of slice for the training step (256 rows per expert) and for MXFP8
    "dsv3_train_slice_e32": LayerShape("dsv3_train_slice_e32", 1024, 7168, 32, 8, 2048, 2048, 1,
                                       0.0, "normal0.1", "bf16", True, 7),
    "dsv3_mxfp8_slice_e32": LayerShape("dsv3_mxfp8_slice_e32", 1024, 7168, 32, 8, 2048, 2048, 1,
                                       0.0, "normal0.1", "mxfp8", False, 8),
    "dsv3_mxfp8_train_slice_e32": LayerShape("dsv3_mxfp8_train_slice_e32", 1024, 7168, 32, 8, 2048,
                                             2048, 1, 0.0, "normal0.1", "mxfp8", True, 11),
    # the DeepSeek-V3 forward with NVFP4 expert GEMMs, and its decode-sized batch
    "dsv3_nvfp4_fwd": LayerShape("dsv3_nvfp4_fwd", 4096, 7168, 256, 8, 2048, 2048, 1, 0.0,
                                 "normal0.1", "nvfp4", False, 13),
    "dsv3_nvfp4_decode_t64": LayerShape("dsv3_nvfp4_decode_t64", 64, 7168, 256, 8, 2048, 2048, 1,
                                        0.0, "normal0.1", "nvfp4", False, 14),
    # the NVFP4 forward on 32 experts with the DSV3 rows per expert (128), for profiler captures
    "dsv3_nvfp4_slice_e32": LayerShape("dsv3_nvfp4_slice_e32", 512, 7168, 32, 8, 2048, 2048, 1, 0.0,
                                       "normal0.1", "nvfp4", False, 15),
    # a slice of the Kimi-class layer for profiler captures: the same rank-biased routing over 48
    # experts (a few hot experts hold nearly every token, CTA-pair tiles), about 4 GB of weights
    "kimi_skew_slice_e48": LayerShape("kimi_skew_slice_e48", 2048, 7168, 48, 8, 2048, 2048, 1, 0.0,
                                      "zipf", "bf16", False, 12),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, seed, device):
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def _stacked_normal(E, rows, cols, std, seed, device):
    """[E,rows,cols] bf16 drawn one expert at a time (bounded temporary memory)."""
    g = _gen(seed, device)
    out = torch.empty((E, rows, cols), dtype=torch.bfloat16, device=device)
    for e in range(E):
        out[e] = (torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def make_layer(shape: LayerShape, device="cpu", with_dy=None, seed_base=None):
    """Draws every input of the layer for ``shape`` on ``device``.  Returns a dict of tensors."""
    c = shape.cid if seed_base is None else seed_base
    T, d, E, F, Fs = shape.T, shape.d, shape.E, shape.F, shape.F_shared
    std_in = shape.weight_std if shape.weight_std > 0 else 1.0 / math.sqrt(d)
    std_f = shape.weight_std if shape.weight_std > 0 else 1.0 / math.sqrt(F)
    std_fs = shape.weight_std if shape.weight_std > 0 else 1.0 / math.sqrt(max(Fs, 1))
    out = {
        "x": _normal((T, d), 1.0, 1000 + c, device),
        "W_router": _normal((d, E), std_in, 2000 + c, device),
        "W_gate": _stacked_normal(E, d, F, std_in, 3000 + c, device),
        "W_up": _stacked_normal(E, d, F, std_in, 4000 + c, device),
        "W_down": _stacked_normal(E, F, d, std_f, 5000 + c, device),
        "bias": None,
        "Ws_gate": None, "Ws_up": None, "Ws_down": None,
    }
    if shape.n_shared:
        out["Ws_gate"] = _normal((d, Fs), std_in, 6000 + c, device)
        out["Ws_up"] = _normal((d, Fs), std_in, 6100 + c, device)
        out["Ws_down"] = _normal((Fs, d), std_fs, 6200 + c, device)
    if shape.bias == "normal0.1":
        g = _gen(7000 + c, device)
        out["bias"] = torch.randn((E,), generator=g, device=device, dtype=torch.float32) * 0.1
    elif shape.bias == "zipf":
        g = _gen(8000 + c, "cpu")
        rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0   # ranks 1..E
        out["bias"] = (1.5 * torch.log(1.0 / rank)).to(torch.float32).to(device)
    if with_dy if with_dy is not None else shape.backward:
        out["dY"] = _normal((T, d), 1.0, 9000 + c, device)
    return out
