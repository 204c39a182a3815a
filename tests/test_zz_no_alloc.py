"""The no-allocation pull schedule (mok_dispatch_index_noalloc) against mok_dispatch_index.

Some callers may not allocate device memory while they route tokens (a runtime that reserves
all of its memory at start-up, or code that must avoid the device-wide synchronisation of
cudaMalloc/cudaFree).  For them the library keeps the counting sort's scratch in its own fixed
device array.  This checks, through the C ABI, that two calls in a row give exactly the outputs
of the workspace entry point (integer outputs: bit-exact), up to the largest size whose histogram
fills the array (T = 65536 at E = 256).  Sizes past it are refused on the host
(tests/test_noalloc_args.py).  The file is collected last on purpose.
"""

import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
from tests._helpers import ensure_lib

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "sorted_tok", "sorted_w", "inv_pos")


def _routing(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    scores = torch.rand((T, E), generator=g)
    scores[:, : E // 4] += 0.5          # skew: some experts hot, some likely empty
    idx = scores.topk(k, dim=1).indices.to(torch.int32)
    w = torch.rand((T, k), generator=g, dtype=torch.float32)
    return idx.cuda(), w.cuda()


def _empty_like_routing(D, dev="cuda"):
    R = D.T * D.k
    return {"counts": torch.full((D.E,), -7, dtype=torch.int32, device=dev),
            "offsets": torch.full((D.E + 1,), -7, dtype=torch.int32, device=dev),
            "sorted_tok": torch.full((R,), -7, dtype=torch.int32, device=dev),
            "sorted_w": torch.full((R,), -7.0, dtype=torch.float32, device=dev),
            "inv_pos": torch.full((D.T, D.k), -7, dtype=torch.int32, device=dev)}


@pytest.mark.parametrize("T,E,k", [(4096, 256, 8), (300, 16, 4), (1, 8, 2), (65536, 256, 8)])
def test_noalloc_matches_workspace_dispatch_twice(T, E, k):
    ensure_lib()
    D = mok.dims(T, 256, E, k, 128, 0, 0)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((T + 1, T + 2)):     # two calls in a row, different routings
        idx, w = _routing(T, E, k, seed)
        want = mok.dispatch_index(D, idx, w, ws)
        got = mok.dispatch_index_noalloc(D, idx, w, _empty_like_routing(D))
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(got[key], want[key]), (call, key)
    assert mok.read_status(ws) == 0
