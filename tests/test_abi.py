"""The C-ABI library loads and exports every symbol include/mok.h declares; host-side argument
checks and size queries behave as documented.  No GPU needed: nothing here launches a kernel."""

import ctypes
import os
import re

import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

import mixture_experts_layer_14_gb300 as mok
from tests._helpers import ROOT, ensure_lib


def _declared():
    with open(os.path.join(ROOT, "include", "mok.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mok_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("mok_route", "mok_dispatch_index", "mok_moe_forward", "mok_moe_backward"):
        assert required in names
    assert sorted(mok.EXPORTED_SYMBOLS) == names


def test_library_exports_every_declared_symbol():
    L = ensure_lib()
    for name in _declared():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {mok.lib_path()}").read()
    for name in _declared():
        assert re.search(rf"\bT {name}\b", out), name


def test_status_strings_and_size_queries():
    L = ensure_lib()
    for code in range(0, -7, -1):
        assert L.mok_status_string(code).decode().startswith("MOK_")
    D = mok.dims(4096, 7168, 256, 8, 2048, 2048, 1)
    fw = mok.workspace_size(D)
    bw = mok.workspace_size(D, backward=True)
    R = 4096 * 8
    assert fw >= 2 * R * 7168 * 2 + R * 2048 * 2          # x_sorted, Y_s and h at least
    assert bw >= 2 * R * 7168 * 2                          # dY_sorted and dX_s at least
    assert mok.saved_size(D) >= 2 * R * 2048 * 2 + R * 7168 * 2   # G, U and x in expert order
    bad = [mok.dims(16, 100, 8, 2, 128), mok.dims(16, 128, 8, 9, 128), mok.dims(16, 128, 12, 2, 128),
           mok.dims(16, 128, 8, 2, 96), mok.dims(-1, 128, 8, 2, 128), mok.dims(16, 128, 1024, 2, 128)]
    for D in bad:
        assert L.mok_workspace_size(ctypes.byref(D), 0) == 0


def test_argument_errors_are_returned_not_raised():
    L = ensure_lib()
    D = mok.dims(16, 128, 8, 2, 128, 128, 1)
    null = None
    # null outputs: MOK_ERR_INVALID_ARG before any CUDA call
    rc = L.mok_route(ctypes.byref(D), null, null, null, null, null, null, null, 0, null)
    assert rc == -1
    rc = L.mok_dispatch_index(ctypes.byref(D), null, null, null, null, null, null, null, null, 0, null)
    assert rc == -1
    # unsupported dims: MOK_ERR_UNSUPPORTED
    Dbad = mok.dims(16, 100, 8, 2, 128, 128, 1)
    rc = L.mok_route(ctypes.byref(Dbad), null, null, null, null, null, null, null, 0, null)
    assert rc == -2
    # misaligned pointer: MOK_ERR_UNSUPPORTED; too-small workspace: MOK_ERR_WORKSPACE
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1001)
    rc = L.mok_route(ctypes.byref(D), odd, fake, null, fake, fake, null, fake, 1 << 40, null)
    assert rc == -2
    rc = L.mok_route(ctypes.byref(D), fake, fake, null, fake, fake, null, fake, 16, null)
    assert rc == -3
    with pytest.raises(mok.MokError):
        mok._check(-3)


def test_mxfp8_backward_sizes_and_argument_errors():
    """MXFP8 training sizes: the backward weight copies (codes + 1/32 scale bytes of the three
    expert weights, routed and shared), the transposed token-axis operands in the backward
    workspace, no x in expert order in `saved`; nothing for bf16; errors returned, not raised,
    with no GPU work."""
    L = ensure_lib()
    T, d, E, k, F, Fs = 8192, 7168, 256, 8, 2048, 2048
    D8 = mok.dims(T, d, E, k, F, Fs, 1, mok.MOK_MXFP8)
    Db = mok.dims(T, d, E, k, F, Fs, 1)
    weights = 3 * (E * d * F + d * Fs)
    pb = L.mok_prepared_bwd_size(ctypes.byref(D8))
    assert weights * (1 + 1 / 32) <= pb <= weights * (1 + 1 / 32) + 12 * 1024
    assert L.mok_prepared_bwd_size(ctypes.byref(Db)) == 0
    R = T * k
    nkb = (R + 127) // 128 + E
    assert mok.workspace_size(D8, backward=True) >= (2 * d + 3 * F) * 128 * nkb   # routed codes
    assert mok.saved_size(D8) < mok.saved_size(Db)          # no bf16 x in expert order
    null = None
    rc = L.mok_prepare_weights_bwd(ctypes.byref(D8), null, null, null)
    assert rc == -1
    W = mok.Weights()
    rc = L.mok_prepare_weights_bwd(ctypes.byref(D8), ctypes.byref(W), null, null)
    assert rc == -1
    rc = L.mok_prepare_weights_bwd(ctypes.byref(Db), ctypes.byref(W), null, null)
    assert rc == 0                                           # bf16: nothing to prepare


def test_plain_c_program_uses_the_abi():
    """tests/c/abi_check.c, a C99 program that includes only mok.h, compiles with -std=c99
    -pedantic -Werror, links against libmok.so and runs its host-side checks (no GPU work)."""
    import shutil
    import subprocess
    import tempfile

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    ensure_lib()
    pkg = os.path.dirname(mok.lib_path())
    cuda_libs = [p for p in ("/usr/local/cuda/lib64", "/usr/local/cuda/lib") if os.path.isdir(p)]
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "abi_check")
        cmd = [gcc, "-std=c99", "-pedantic", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
               os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe, mok.lib_path(),
               "-Wl,-rpath," + pkg, "-Wl,--allow-shlib-undefined"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        env = dict(os.environ)
        env["LD_LIBRARY_PATH"] = ":".join(cuda_libs + [pkg, env.get("LD_LIBRARY_PATH", "")])
        r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=60)
        assert r.returncode == 0 and "abi_check ok" in r.stdout, r.stdout + r.stderr


def test_forward_schedule_values():
    """The process-wide forward schedule takes its two values and refuses others (host only)."""
    mok.lib()
    prev = mok.set_forward_schedule(mok.SCHEDULE_FUSED)
    try:
        assert mok.set_forward_schedule(mok.SCHEDULE_TWO_LAUNCHES) == mok.SCHEDULE_FUSED
        with pytest.raises(mok.MokError):
            mok.set_forward_schedule(7)
    finally:
        mok.set_forward_schedule(prev)


def test_nvfp4_sizes_and_argument_errors():
    """NVFP4 prepared size (codes 1/2 byte and scales 1/16 byte per weight element, plus the
    per-matrix scales and the two calibration values); no saved activations (forward only); the
    backward and invalid calibration values are refused on the host, before any CUDA call."""
    L = ensure_lib()
    E, d, F, Fs = 256, 7168, 2048, 2048
    D = mok.dims(4096, d, E, 8, F, Fs, 1, dtype=mok.MOK_NVFP4)
    elems = 3 * E * d * F + 3 * d * Fs
    n = mok.prepared_size(D)
    assert elems * 9 // 16 <= n <= elems * 9 // 16 + 16 * 1024 + 8 * (3 * E + 3) + 1024
    assert mok.saved_size(D) == 0
    assert mok.prepared_size(mok.dims(16, 128, 8, 2, 128, 128, 1, dtype=mok.MOK_NVFP4)) == 0  # d % 256
    null = None
    fake = ctypes.c_void_p(0x1000)
    f = ctypes.c_float
    Dn = mok.dims(16, 256, 8, 2, 128, 128, 1, dtype=mok.MOK_NVFP4)
    Db = mok.dims(16, 256, 8, 2, 128, 128, 1)
    set_amax = L.mok_nvfp4_set_activation_amax
    assert set_amax(ctypes.byref(Db), fake, f(1.0), f(1.0), null) == -1      # not NVFP4
    assert set_amax(ctypes.byref(Dn), null, f(1.0), f(1.0), null) == -1      # no buffer
    assert set_amax(ctypes.byref(Dn), ctypes.c_void_p(0x1001), f(1.0), f(1.0), null) == -1
    assert set_amax(ctypes.byref(Dn), fake, f(-1.0), f(1.0), null) == -1
    assert set_amax(ctypes.byref(Dn), fake, f(1.0), f(float("nan")), null) == -1
    assert set_amax(ctypes.byref(Dn), fake, f(float("inf")), f(1.0), null) == -1
    rc = L.mok_moe_backward(ctypes.byref(Dn), *([null] * 20), 0, null)
    assert rc == -2
