"""MXFP8 block quantisation, written from the format definitions.  Test infrastructure only.

Format (the MXFP8 path of the layer; pages: "Mixture-of-Kittens; MoE megakernel", key points —
BF16 and MXFP8 supported): E4M3 values ("fn" variant: bias 7, no infinities, S.1111.111 is NaN,
largest finite 448) with one UE8M0 power-of-two scale per 32 contiguous elements along the
reduction dimension.  The scale of a block is its amax / 448 rounded up to a power of two, i.e.
2^s with s the smallest integer such that amax <= 448 * 2^s (s clamped to [-127, 127]; an all-zero
block takes s = -127, byte 0x00).  Values are divided by the scale and rounded to the nearest
E4M3 value, ties to an even mantissa, saturating to +-448.

Pins (tests): all 256 codes decode/encode round trip; bit-exact agreement with the
torch.float8_e4m3fn conversion routine on random and edge values; the scale rule on blocks whose
amax is exactly 448 * 2^s and just above it.
"""

import numpy as np

E4M3_MAX = 448.0
MX_BLOCK = 32


def e4m3_decode(codes):
    """Value of each E4M3 code (uint8 array) as float64; NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode(v):
    """Nearest E4M3 code of each float64 value: round to nearest with ties to an even mantissa,
    saturating to +-448 (NaN -> 0x7F with the sign bit of the input).

    The E4M3 grid in the binade [2^(e-1), 2^e) has 8 steps of 2^(e-4) for e-1 >= -6 and steps of
    2^-9 below 2^-6 (subnormals); the value is divided by its step (exact power of two), rounded
    to an integer with ties to even (np.rint), and multiplied back.  An even step count is an even
    mantissa, so ties go to the even code."""
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    a = np.where(nan, 0.0, np.minimum(np.abs(v), E4M3_MAX))
    _, e = np.frexp(a)                                   # a = m 2^e, m in [0.5, 1)
    step = np.maximum(e - 1, -6) - 3                     # exponent of the grid step
    q = np.rint(np.ldexp(a, -step))                      # steps, ties to even
    val = np.ldexp(q, step)                              # the rounded magnitude (exact)
    # fields of the rounded magnitude
    m2, e2 = np.frexp(val)
    normal = val >= 2.0 ** -6
    E = np.where(normal, e2 + 6, 0)
    M = np.where(normal, np.rint((2.0 * m2 - 1.0) * 8.0), np.rint(np.ldexp(val, 9)))
    code = (E.astype(np.int64) << 3) | M.astype(np.int64)
    code = np.where(nan, 0x7F, code).astype(np.uint8)
    return np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)


def mx_scale_exponent(amax):
    """Smallest integer s in [-127, 127] with amax <= 448 * 2^s (exact comparisons)."""
    a = np.asarray(amax, dtype=np.float64)
    safe = np.where(a > 0, a, 1.0)
    s = np.ceil(np.log2(safe / E4M3_MAX))
    # correct any rounding of log2 with exact power-of-two comparisons
    s = np.where(E4M3_MAX * np.exp2(s - 1) >= safe, s - 1, s)
    s = np.where(E4M3_MAX * np.exp2(s) < safe, s + 1, s)
    s = np.where(a > 0, s, -127.0)
    return np.clip(s, -127, 127).astype(np.int64)


def mx_quantize(v):
    """Quantise v[..., K] (K a multiple of 32) along its last axis.  Returns (codes uint8
    [..., K], scale bytes uint8 [..., K/32]) where the scale byte is s + 127."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % MX_BLOCK == 0
    blocks = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    s = mx_scale_exponent(np.abs(blocks).max(axis=-1))
    q = e4m3_encode(np.ldexp(blocks, -s[..., None]))
    return q.reshape(v.shape), (s + 127).astype(np.uint8)


_DECODE_TABLE = e4m3_decode(np.arange(256, dtype=np.uint8))  # the 256 code values, once


def mx_dequantize(codes, scale_bytes):
    """codes[..., K] * 2^(scale_byte - 127) per block of 32, float64."""
    c = np.asarray(codes, dtype=np.uint8)
    K = c.shape[-1]
    vals = _DECODE_TABLE[c].reshape(c.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    s = np.asarray(scale_bytes, dtype=np.int64) - 127
    return np.ldexp(vals, s[..., None]).reshape(c.shape)
