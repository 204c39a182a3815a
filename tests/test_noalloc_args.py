"""Host-side argument checks of the no-allocation pull schedule, on the CPU.

The binding checks every tensor before it hands raw pointers to the library (a wrong dtype,
shape or device would otherwise let the kernels read or write out of bounds), and the library
refuses sizes whose histogram does not fit its fixed scratch array before it touches the GPU.
"""

import ctypes

import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
from tests._helpers import ensure_lib


def _inputs(T=40, E=16, k=4, dev="cpu"):
    R = T * k
    idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    out = {"counts": torch.empty((E,), dtype=torch.int32, device=dev),
           "offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
           "sorted_tok": torch.empty((R,), dtype=torch.int32, device=dev),
           "sorted_w": torch.empty((R,), dtype=torch.float32, device=dev),
           "inv_pos": torch.empty((T, k), dtype=torch.int32, device=dev)}
    return mok.dims(T, 256, E, k, 128, 0, 0), idx, w, out


def test_wrong_dtype_shape_or_device_raise_before_any_call():
    D, idx, w, out = _inputs()
    with pytest.raises(ValueError, match="topk_idx: dtype"):
        mok.dispatch_index_noalloc(D, idx.to(torch.int64), w, out)
    with pytest.raises(ValueError, match="topk_w: shape"):
        mok.dispatch_index_noalloc(D, idx, w[:, :2], out)
    bad = dict(out, sorted_tok=out["sorted_tok"][:-1])          # one destination row short
    with pytest.raises(ValueError, match="sorted_tok.*shape"):
        mok.dispatch_index_noalloc(D, idx, w, bad)
    bad = dict(out, offsets=out["offsets"].to(torch.int64))
    with pytest.raises(ValueError, match="offsets.*dtype"):
        mok.dispatch_index_noalloc(D, idx, w, bad)
    bad = dict(out)
    del bad["inv_pos"]
    with pytest.raises(ValueError, match="inv_pos.*required"):
        mok.dispatch_index_noalloc(D, idx, w, bad)
    with pytest.raises(ValueError, match="must live on"):        # host tensors, right shapes
        mok.dispatch_index_noalloc(D, idx, w, out)


@pytest.mark.parametrize("T,E", [(65536 + 64, 256), (32768 + 64, 512), (64 * 600, 512)])
def test_sizes_past_the_scratch_are_refused(T, E):
    """E * ceil(T / 64) histogram counts must fit in 262144 words: one 64-token chunk past the
    limit is refused with MOK_ERR_WORKSPACE before any CUDA call (fake pointers are never
    touched)."""
    L = ensure_lib()
    D = mok.dims(T, 256, E, 8, 128, 0, 0)
    fake = ctypes.c_void_p(0x1000)
    rc = L.mok_dispatch_index_noalloc(ctypes.byref(D), fake, fake, fake, fake, fake, fake, fake, None)
    assert rc == -3

