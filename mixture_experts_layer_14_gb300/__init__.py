"""GB300-native (sm_103a) DeepSeek-V3-style MoE layer — Python binding of the C-ABI library.

This module only marshals arguments: it checks tensor shapes, dtypes, devices and contiguity,
allocates outputs with PyTorch and passes raw device pointers and the current CUDA stream to
``libmok.so`` (declared in ``include/mok.h``).  Every step of the layer runs in that library's
kernels.  There is no fallback: without the compiled library every call raises.

Entry points mirror the C ABI: :func:`route`, :func:`dispatch_index`, :func:`moe_forward`,
:func:`moe_backward`, :func:`layer_forward_host`, plus :class:`MoELayer`, a small convenience
holder of weights and workspaces.
"""

import ctypes
import os

import torch

__all__ = [
    "MokError", "Dims", "Weights", "lib", "lib_path", "dims", "route", "dispatch_index",
    "moe_forward", "moe_backward", "layer_forward_host", "workspace_size", "saved_size",
    "read_status", "clear_status", "last_launch_count", "MoELayer", "EXPORTED_SYMBOLS",
    "MOK_BF16", "MOK_MXFP8", "MOK_NVFP4", "prepare_weights", "prepare_weights_bwd",
    "mx_quantize_rows", "nvfp4_set_activation_amax",
]

MOK_BF16, MOK_MXFP8, MOK_NVFP4 = 0, 1, 2
PASS_FORWARD, PASS_BACKWARD = 0, 1

EXPORTED_SYMBOLS = [
    "mok_workspace_size", "mok_saved_size", "mok_prepared_size", "mok_prepare_weights",
    "mok_route", "mok_dispatch_index", "mok_moe_forward", "mok_moe_backward",
    "mok_layer_host_extra_size", "mok_layer_forward_host", "mok_status_string",
    "mok_read_device_status", "mok_clear_device_status", "mok_last_launch_count",
    "mok_timing_enable", "mok_timing_collect", "mok_dispatch_index_noalloc",
    "mok_mx_quantize_rows", "mok_selftest_bounded_wait", "mok_prepared_bwd_size",
    "mok_prepare_weights_bwd", "mok_set_forward_schedule", "mok_nvfp4_set_activation_amax",
]


class MokError(RuntimeError):
    pass


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("F_shared", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "W_router", "router_bias", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down",
        "prepared", "prepared_bwd")]


_LIB = None
_VP = ctypes.c_void_p
_SZ = ctypes.c_size_t
_DP = ctypes.POINTER(Dims)
_WP = ctypes.POINTER(Weights)


def lib_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmok.so")


def lib():
    """The loaded libmok.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise MokError(f"{path} is missing; build it with `python -m mixture_experts_layer_14_gb300.build`")
        L = ctypes.CDLL(path)
        sig = {
            "mok_workspace_size": (_SZ, [_DP, ctypes.c_int]),
            "mok_saved_size": (_SZ, [_DP]),
            "mok_prepared_size": (_SZ, [_DP]),
            "mok_prepared_bwd_size": (_SZ, [_DP]),
            "mok_prepare_weights_bwd": (ctypes.c_int, [_DP, _WP, _VP, _VP]),
            "mok_layer_host_extra_size": (_SZ, [_DP]),
            "mok_prepare_weights": (ctypes.c_int, [_DP, _WP, _VP, _VP]),
            "mok_route": (ctypes.c_int, [_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
            "mok_dispatch_index": (ctypes.c_int, [_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
            "mok_moe_forward": (ctypes.c_int, [_DP, _WP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
            "mok_moe_backward": (ctypes.c_int, [_DP, _WP] + [_VP] * 19 + [_SZ, _VP]),
            "mok_layer_forward_host": (ctypes.c_int, [_DP, _WP, _VP, _VP, _VP, _SZ, _VP]),
            "mok_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "mok_read_device_status": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int), _VP]),
            "mok_clear_device_status": (ctypes.c_int, [_VP, _VP]),
            "mok_last_launch_count": (ctypes.c_int, []),
            "mok_timing_enable": (ctypes.c_int, [ctypes.c_int]),
            "mok_selftest_bounded_wait": (ctypes.c_int, [_VP, ctypes.c_int64, _VP]),
            "mok_mx_quantize_rows": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, _VP, _VP, _VP, _VP]),
            "mok_dispatch_index_noalloc": (ctypes.c_int, [_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
            "mok_set_forward_schedule": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
            "mok_nvfp4_set_activation_amax": (ctypes.c_int, [_DP, _VP, ctypes.c_float, ctypes.c_float, _VP]),
            "mok_timing_collect": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_int),
                                                  ctypes.POINTER(ctypes.c_double), ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_int)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(rc):
    if rc != 0:
        raise MokError(lib().mok_status_string(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _want(t, name, shape, dtype, device, check_device=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if check_device and (not t.is_cuda or (device is not None and t.device != device)):
        raise ValueError(f"{name} must live on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def dims(T, d, E, k, F, F_shared=0, n_shared=1, dtype=MOK_BF16):
    return Dims(T, d, E, k, F, F_shared if n_shared else 0, n_shared, dtype)


def workspace_size(D, backward=False):
    n = lib().mok_workspace_size(ctypes.byref(D), PASS_BACKWARD if backward else PASS_FORWARD)
    if n == 0:
        raise MokError("unsupported layer dimensions")
    return n


def saved_size(D):
    return lib().mok_saved_size(ctypes.byref(D))


def read_status(ws):
    v = ctypes.c_int(0)
    _check(lib().mok_read_device_status(_ptr(ws), ctypes.byref(v), _stream()))
    return v.value


def clear_status(ws):
    _check(lib().mok_clear_device_status(_ptr(ws), _stream()))


def last_launch_count():
    return lib().mok_last_launch_count()


def selftest_bounded_wait(ws, budget_ns=50_000_000):
    """Runs a kernel whose bounded wait must run out; the status word of ws then reads
    MOK_ERR_TIMEOUT (-5)."""
    _check(lib().mok_selftest_bounded_wait(_ptr(ws), int(budget_ns), _stream()))


SCHEDULE_TWO_LAUNCHES, SCHEDULE_FUSED = 0, 1


def set_forward_schedule(schedule):
    """Process-wide schedule of the bf16 forward's expert GEMMs (SCHEDULE_TWO_LAUNCHES, the
    default, or SCHEDULE_FUSED: one persistent launch fed by a device work counter); returns the
    previous one.  Results are bit-identical under both."""
    prev = ctypes.c_int(0)
    _check(lib().mok_set_forward_schedule(int(schedule), ctypes.byref(prev)))
    return prev.value


def timing_enable(on=True):
    """Record a CUDA event pair around every kernel the library launches on this thread."""
    _check(lib().mok_timing_enable(1 if on else 0))


def timing_collect(max_kernels=64):
    """{kernel name: (launches, summed device ms)} of the recorded launches; clears them."""
    names = ctypes.create_string_buffer(32 * max_kernels)
    launches = (ctypes.c_int * max_kernels)()
    ms = (ctypes.c_double * max_kernels)()
    n = ctypes.c_int(0)
    _check(lib().mok_timing_collect(names, launches, ms, max_kernels, ctypes.byref(n)))
    out = {}
    for i in range(n.value):
        name = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
        out[name] = (launches[i], ms[i])
    return out


def _weights_struct(D, W):
    dev = W["W_gate"].device
    bf = torch.bfloat16
    _want(W["W_router"], "W_router", (D.d, D.E), bf, dev)
    _want(W["W_gate"], "W_gate", (D.E, D.d, D.F), bf, dev)
    _want(W["W_up"], "W_up", (D.E, D.d, D.F), bf, dev)
    _want(W["W_down"], "W_down", (D.E, D.F, D.d), bf, dev)
    if W.get("bias") is not None:
        _want(W["bias"], "bias", (D.E,), torch.float32, dev)
    if D.n_shared:
        _want(W["Ws_gate"], "Ws_gate", (D.d, D.F_shared), bf, dev)
        _want(W["Ws_up"], "Ws_up", (D.d, D.F_shared), bf, dev)
        _want(W["Ws_down"], "Ws_down", (D.F_shared, D.d), bf, dev)
    return Weights(
        W["W_router"].data_ptr(), W["bias"].data_ptr() if W.get("bias") is not None else None,
        W["W_gate"].data_ptr(), W["W_up"].data_ptr(), W["W_down"].data_ptr(),
        W["Ws_gate"].data_ptr() if D.n_shared else None,
        W["Ws_up"].data_ptr() if D.n_shared else None,
        W["Ws_down"].data_ptr() if D.n_shared else None,
        W["prepared"].data_ptr() if W.get("prepared") is not None else None,
        W["prepared_bwd"].data_ptr() if W.get("prepared_bwd") is not None else None)


def route(D, x, W_router, bias, ws, want_logits=False):
    """Returns (topk_idx[T,k] int32, topk_w[T,k] fp32, logits[T,E] fp32 or None)."""
    dev = x.device
    _want(x, "x", (D.T, D.d), torch.bfloat16, dev)
    _want(W_router, "W_router", (D.d, D.E), torch.bfloat16, dev)
    if bias is not None:
        _want(bias, "bias", (D.E,), torch.float32, dev)
    idx = torch.empty((D.T, D.k), dtype=torch.int32, device=dev)
    w = torch.empty((D.T, D.k), dtype=torch.float32, device=dev)
    logits = torch.empty((D.T, D.E), dtype=torch.float32, device=dev) if want_logits else None
    _check(lib().mok_route(ctypes.byref(D), _ptr(x), _ptr(W_router), _ptr(bias), _ptr(idx), _ptr(w),
                           _ptr(logits), _ptr(ws), ws.numel(), _stream()))
    return idx, w, logits


def dispatch_index(D, topk_idx, topk_w, ws):
    """Returns a dict with counts[E], offsets[E+1], sorted_tok[T*k], sorted_w[T*k], inv_pos[T,k]."""
    dev = topk_idx.device
    _want(topk_idx, "topk_idx", (D.T, D.k), torch.int32, dev)
    _want(topk_w, "topk_w", (D.T, D.k), torch.float32, dev)
    R = D.T * D.k
    out = {
        "topk_idx": topk_idx, "topk_w": topk_w,
        "counts": torch.empty((D.E,), dtype=torch.int32, device=dev),
        "offsets": torch.empty((D.E + 1,), dtype=torch.int32, device=dev),
        "sorted_tok": torch.empty((R,), dtype=torch.int32, device=dev),
        "sorted_w": torch.empty((R,), dtype=torch.float32, device=dev),
        "inv_pos": torch.empty((D.T, D.k), dtype=torch.int32, device=dev),
    }
    _check(lib().mok_dispatch_index(
        ctypes.byref(D), _ptr(topk_idx), _ptr(topk_w), _ptr(out["counts"]), _ptr(out["offsets"]),
        _ptr(out["sorted_tok"]), _ptr(out["sorted_w"]), _ptr(out["inv_pos"]), _ptr(ws), ws.numel(),
        _stream()))
    return out


def dispatch_index_noalloc(D, topk_idx, topk_w, out):
    """Pull schedule into the caller's preallocated tensors ``out`` (same keys as the dict of
    :func:`dispatch_index`) without a workspace: for callers that may not allocate device memory
    while routing.  The library keeps its scratch in a fixed device array (1 MiB of histogram),
    looked up for the current device, so every tensor must live there."""
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cuda"
    R = D.T * D.k
    specs = [(topk_idx, "topk_idx", (D.T, D.k), torch.int32), (topk_w, "topk_w", (D.T, D.k), torch.float32)]
    for key, shape, dtype in (("counts", (D.E,), torch.int32), ("offsets", (D.E + 1,), torch.int32),
                              ("sorted_tok", (R,), torch.int32), ("sorted_w", (R,), torch.float32),
                              ("inv_pos", (D.T, D.k), torch.int32)):
        specs.append((out.get(key), f"out[{key!r}]", shape, dtype))
    for t, name, shape, dtype in specs:      # every shape and dtype first, then the devices
        _want(t, name, shape, dtype, None, check_device=False)
    for t, name, shape, dtype in specs:
        _want(t, name, shape, dtype, dev)
    _check(lib().mok_dispatch_index_noalloc(
        ctypes.byref(D), _ptr(topk_idx), _ptr(topk_w), _ptr(out["counts"]), _ptr(out["offsets"]),
        _ptr(out["sorted_tok"]), _ptr(out["sorted_w"]), _ptr(out["inv_pos"]), _stream()))
    return out


def mx_quantize_rows(src):
    """MXFP8 quantisation of a [rows, K] bf16 CUDA tensor along K: (codes uint8 [rows, K],
    UE8M0 scale bytes uint8 [rows, K/32])."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous() or src.dim() != 2:
        raise ValueError("src must be a contiguous 2-D bf16 CUDA tensor")
    rows, K = src.shape
    q = torch.empty((rows, K), dtype=torch.uint8, device=src.device)
    sc = torch.empty((rows, K // 32), dtype=torch.uint8, device=src.device)
    _check(lib().mok_mx_quantize_rows(rows, K, _ptr(src), _ptr(q), _ptr(sc), _stream()))
    return q, sc


def prepared_size(D):
    return lib().mok_prepared_size(ctypes.byref(D))


def prepare_weights(D, W):
    """MXFP8 / NVFP4: quantised copy of the expert weights in the layout of mok_prepare_weights
    (uint8 CUDA tensor); returns None for bf16.  Pass it as W["prepared"].  NVFP4: set the
    calibrated activation amaxes with :func:`nvfp4_set_activation_amax` afterwards."""
    n = prepared_size(D)
    if n == 0:
        return None
    buf = torch.empty(n, dtype=torch.uint8, device=W["W_gate"].device)
    Wd = dict(W)
    Wd["prepared"] = None
    Wd["prepared_bwd"] = None
    st = _weights_struct(D, Wd)
    _check(lib().mok_prepare_weights(ctypes.byref(D), ctypes.byref(st), _ptr(buf), _stream()))
    return buf


def nvfp4_set_activation_amax(D, prepared, amax_x, amax_h):
    """NVFP4: the calibrated tensor amaxes of x and h, written into ``prepared``."""
    _want(prepared, "prepared", (prepared_size(D),), torch.uint8, prepared.device)
    _check(lib().mok_nvfp4_set_activation_amax(ctypes.byref(D), _ptr(prepared), float(amax_x),
                                                float(amax_h), _stream()))


def prepare_weights_bwd(D, W):
    """MXFP8: the expert weights quantised along the backward GEMMs' reduction dimensions (uint8
    CUDA tensor); returns None for bf16.  Pass it as W["prepared_bwd"] for the MXFP8 backward."""
    n = lib().mok_prepared_bwd_size(ctypes.byref(D))
    if n == 0:
        return None
    buf = torch.empty(n, dtype=torch.uint8, device=W["W_gate"].device)
    Wd = dict(W)
    Wd["prepared"] = None
    Wd["prepared_bwd"] = None
    st = _weights_struct(D, Wd)
    _check(lib().mok_prepare_weights_bwd(ctypes.byref(D), ctypes.byref(st), _ptr(buf), _stream()))
    return buf


def moe_forward(D, W, x, routing, ws, saved=None, y=None):
    """y[T,d] bf16 of the expert part for a routing from :func:`dispatch_index`."""
    dev = x.device
    _want(x, "x", (D.T, D.d), torch.bfloat16, dev)
    ws_struct = _weights_struct(D, W)
    if y is None:
        y = torch.empty((D.T, D.d), dtype=torch.bfloat16, device=dev)
    _check(lib().mok_moe_forward(
        ctypes.byref(D), ctypes.byref(ws_struct), _ptr(x), _ptr(routing["topk_idx"]),
        _ptr(routing["offsets"]), _ptr(routing["sorted_tok"]), _ptr(routing["sorted_w"]),
        _ptr(routing["inv_pos"]), _ptr(y), _ptr(saved), _ptr(ws), ws.numel(), _stream()))
    return y


def moe_backward(D, W, x, dY, saved, routing, ws, want_dW_router=True):
    """Gradients of the layer for upstream dY (selection held constant).  Returns a dict."""
    dev = x.device
    bf = torch.bfloat16
    _want(dY, "dY", (D.T, D.d), bf, dev)
    ws_struct = _weights_struct(D, W)
    g = {
        "dX": torch.empty((D.T, D.d), dtype=bf, device=dev),
        "dW_gate": torch.empty((D.E, D.d, D.F), dtype=bf, device=dev),
        "dW_up": torch.empty((D.E, D.d, D.F), dtype=bf, device=dev),
        "dW_down": torch.empty((D.E, D.F, D.d), dtype=bf, device=dev),
        "dWs_gate": torch.empty((D.d, D.F_shared), dtype=bf, device=dev) if D.n_shared else None,
        "dWs_up": torch.empty((D.d, D.F_shared), dtype=bf, device=dev) if D.n_shared else None,
        "dWs_down": torch.empty((D.F_shared, D.d), dtype=bf, device=dev) if D.n_shared else None,
        "dlogits": torch.empty((D.T, D.E), dtype=torch.float32, device=dev),
        "dW_router": torch.empty((D.d, D.E), dtype=bf, device=dev) if want_dW_router else None,
    }
    r = routing
    _check(lib().mok_moe_backward(
        ctypes.byref(D), ctypes.byref(ws_struct), _ptr(x), _ptr(dY), _ptr(saved), _ptr(r["topk_idx"]),
        _ptr(r["topk_w"]), _ptr(r["offsets"]), _ptr(r["sorted_tok"]), _ptr(r["sorted_w"]),
        _ptr(r["inv_pos"]), _ptr(g["dX"]), _ptr(g["dW_gate"]), _ptr(g["dW_up"]), _ptr(g["dW_down"]),
        _ptr(g["dWs_gate"]), _ptr(g["dWs_up"]), _ptr(g["dWs_down"]), _ptr(g["dlogits"]),
        _ptr(g["dW_router"]), _ptr(ws), ws.numel(), _stream()))
    return g


def layer_forward_host(D, W, x_host, y_host, ws):
    """Whole-layer forward with x and y in (pinned) host memory; asynchronous on the current
    stream.  ``ws`` must hold workspace_size(D) + host_extra_size(D) bytes."""
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("x_host and y_host must be host tensors")
    ws_struct = _weights_struct(D, W)
    _check(lib().mok_layer_forward_host(ctypes.byref(D), ctypes.byref(ws_struct), _ptr(x_host),
                                        _ptr(y_host), _ptr(ws), ws.numel(), _stream()))


def host_extra_size(D):
    return lib().mok_layer_host_extra_size(ctypes.byref(D))


class MoELayer:
    """Holds the weights of one layer and its workspaces; calls the C ABI in sequence."""

    def __init__(self, D, W, device=None):
        self.D = D
        self.W = W
        dev = device or W["W_gate"].device
        self.ws = torch.zeros(workspace_size(D), dtype=torch.uint8, device=dev)
        self.saved = None
        self._ws_bwd = None

    def forward(self, x, training=False):
        idx, w, _ = route(self.D, x, self.W["W_router"], self.W.get("bias"), self.ws)
        n = last_launch_count()
        routing = dispatch_index(self.D, idx, w, self.ws)
        n += last_launch_count()
        if training and self.saved is None:
            self.saved = torch.empty(saved_size(self.D), dtype=torch.uint8, device=x.device)
        y = moe_forward(self.D, self.W, x, routing, self.ws, saved=self.saved if training else None)
        self.last_launches = n + last_launch_count()  # kernels this call enqueued
        self.routing = routing
        return y

    def backward(self, x, dY):
        if self._ws_bwd is None:
            self._ws_bwd = torch.zeros(workspace_size(self.D, backward=True), dtype=torch.uint8,
                                       device=x.device)
        g = moe_backward(self.D, self.W, x, dY, self.saved, self.routing, self._ws_bwd)
        self.last_launches = last_launch_count()
        return g
