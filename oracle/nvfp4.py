"""NVFP4 block quantisation, written from the format definition.  Test infrastructure only.

The pages name NVFP4 only as the format of their authors' earlier training kernels (page
"Mixture-of-Kittens: Nhân kernel MoE nguồn mở tối ưu cho hệ thống NVL72", opening section on the
team's prior MXFP8 and NVFP4 kernels); they define neither the format nor a recipe.  The format
is NVIDIA's NVFP4:
  * elements E2M1: a sign bit, two exponent bits (bias 1) and one mantissa bit; magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN.  Code = sign << 3 | magnitude index.
  * one E4M3 scale (positive) per 16 consecutive elements along the reduction dimension;
  * one fp32 scale per tensor, so that the block scales stay inside E4M3's range.

Reading of the recipe (the plain two-level one; every step in fp32, each operation rounded to
the nearest fp32 with ties to even, so that a kernel can take the same decisions bit for bit):
  A = the tensor's amax (for activations: a calibrated value given with the layer);
  S = 2688 / A (2688 = 6 * 448: the largest block amax maps onto the largest scale times the
      largest element); S = 1 when A is 0;
  per block of 16:  s = E4M3_rn((a / 6) * S), a = the block's amax (saturating at 448);
  per element:      q = E2M1_rn(v * (S / s_val)), ties to an even code (even magnitude index),
                    saturating to +-6; q = 0 when s_val is 0; the sign bit is set when
                    v * (S / s_val) < 0;
  value = q_val * s_val * g with g = 1 / S (fp32): the GEMM multiplies q_val * s_val products
  and applies the two tensors' g in its epilogue.

Pins (tests/test_oracle_nvfp4.py): all 16 codes; E2M1 rounding against a brute-force nearest
search with ties to the even code; saturation; the scale rule's closed forms; fixed points
(values q_val * s_val * g round-trip exactly); the block and tensor-scale axes; invariance of the
codes under power-of-two scaling of a tensor.
"""

import numpy as np

from .mxfp8 import e4m3_decode, e4m3_encode

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
NV_BLOCK = 16
NV_RANGE = 6.0 * 448.0  # 2688


def e2m1_decode(codes):
    """Value of each E2M1 code (uint8 array holding one code per element, low nibble)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = E2M1_VALUES[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e2m1_encode(v):
    """Nearest E2M1 code of each float64 value: the magnitude grid has steps of 0.5 below 2, 1
    in [2, 4) and 2 in [4, 6]; the magnitude is divided by its step (a power of two), rounded to
    an integer with ties to even (np.rint) and multiplied back, then saturated at 6.  An even
    number of steps is an even magnitude index, so ties go to the even code.  Sign bit: v < 0."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.rint(a / step) * step, 6.0)
    idx = np.searchsorted(E2M1_VALUES, r)           # r is exactly one of the grid values
    return (idx | np.where(v < 0, 8, 0)).astype(np.uint8)


def nv_tensor_scale(amax):
    """S = 2688 / A in fp32 (1 when A is 0) and the decode scale g = 1 / S in fp32."""
    A = np.float32(amax)
    S = np.float32(NV_RANGE) / A if A > 0 else np.float32(1.0)
    return np.float32(S), np.float32(np.float32(1.0) / S)


def nv_quantize(v, tensor_amax=None):
    """Quantise v[..., K] (K a multiple of 16) along its last axis.  The values are first
    rounded to fp32 (exact for bf16 inputs).  ``tensor_amax``: the tensor's A (default: max |v|).
    Returns (codes uint8 [..., K], scale codes uint8 [..., K/16], g fp32)."""
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    K = v32.shape[-1]
    assert K % NV_BLOCK == 0
    A = np.abs(v32).max() if tensor_amax is None else tensor_amax
    S, g = nv_tensor_scale(A)
    blocks = v32.reshape(v32.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    a = np.abs(blocks).max(axis=-1)
    u = (a / np.float32(6.0)) * S                               # fp32, two roundings
    sc = e4m3_encode(u.astype(np.float64))                     # nearest, saturating at 448
    sv = e4m3_decode(sc).astype(np.float32)
    inv = np.where(sv > 0, S / np.where(sv > 0, sv, np.float32(1.0)), np.float32(0.0))
    t = blocks * inv.astype(np.float32)[..., None]             # fp32
    q = e2m1_encode(t.astype(np.float64))
    return q.reshape(v32.shape), sc.astype(np.uint8), g


def nv_dequantize(codes, scale_codes, g):
    """codes[..., K] values * their block's scale * g, float64 (every product exact)."""
    c = np.asarray(codes, dtype=np.uint8)
    K = c.shape[-1]
    vals = e2m1_decode(c).reshape(c.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    s = e4m3_decode(np.asarray(scale_codes, dtype=np.uint8))
    return (vals * s[..., None] * np.float64(g)).reshape(c.shape)
