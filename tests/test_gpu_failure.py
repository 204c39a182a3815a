"""Failure detection on the GPU without a fault: a kernel wait that nothing satisfies gives up
after its budget, records MOK_ERR_TIMEOUT in the status word and returns; the context stays
usable and the next layer call is correct."""

import pytest
import torch

import mixture_experts_layer_14_gb300 as mok
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS, make_layer
from tests._helpers import dims_of, ensure_lib, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ensure_lib()
    shape = WORKLOADS["tiny"]
    D = dims_of(shape)
    ws = torch.zeros(mok.workspace_size(D), dtype=torch.uint8, device="cuda")
    assert mok.read_status(ws) == 0
    mok.selftest_bounded_wait(ws, budget_ns=50_000_000)  # 50 ms
    assert mok.read_status(ws) == -5  # MOK_ERR_TIMEOUT
    mok.clear_status(ws)
    assert mok.read_status(ws) == 0
    # the context still works: a full forward runs and reports no error
    L = to_dev(make_layer(shape, "cpu"))
    layer = mok.MoELayer(D, L)
    y = layer.forward(L["x"])
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all() and mok.read_status(layer.ws) == 0


def test_selftest_rejects_bad_budgets():
    L = ensure_lib()
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    import ctypes
    assert L.mok_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 0, None) == -1
    assert L.mok_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 10**10, None) == -1
