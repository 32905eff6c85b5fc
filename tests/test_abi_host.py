"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function that include/fbob.h
declares, and argument validation must reject bad calls before touching the
GPU (no CUDA call happens on these paths, so they run without a device).
"""

import ctypes
import os
import re
import subprocess

import pytest

import exact_second_order_attn_gb300 as fb
from exact_second_order_attn_gb300 import _lib
from exact_second_order_attn_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fbob.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fbob_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("fbob_attn_fwd", "fbob_attn_bwd", "fbob_attn_bob", "fbob_bob_workspace_bytes"):
        assert n in names


def test_library_exports_every_header_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fb.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        getattr(lib, name)
    assert set(_lib.FUNCTIONS) <= set(header_functions())


def test_abi_version_and_status_strings(lib):
    assert lib.fbob_abi_version() == 1
    for code, name in enumerate(["FBOB_OK", "FBOB_ERR_INVALID_ARG", "FBOB_ERR_UNSUPPORTED",
                                 "FBOB_ERR_WORKSPACE", "FBOB_ERR_CUDA", "FBOB_ERR_TIMEOUT"]):
        assert lib.fbob_status_string(code).decode() == name


def test_workspace_bytes(lib):
    p = _lib.Problem(2, 3, 256, 64, 0.125, _lib.BF16, 0)
    assert lib.fbob_bob_workspace_bytes(ctypes.byref(p)) == 2 * 4 * 2 * 3 * 256
    assert lib.fbob_bob_workspace_bytes(None) == 0


def fake(addr):
    return ctypes.c_void_p(addr)


def call_bob(lib, p, ptrs=None, ws=0x10000, ws_bytes=None):
    ptrs = ptrs or [0x1000 * (k + 1) for k in range(14)]
    if ws_bytes is None:
        ws_bytes = lib.fbob_bob_workspace_bytes(ctypes.byref(p))
    args = [fake(x) for x in ptrs]
    return lib.fbob_attn_bob(ctypes.byref(p), *args, fake(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("field,value,status", [
    ("d", 48, _lib.ERR_UNSUPPORTED),
    ("d", 256, _lib.ERR_UNSUPPORTED),
    ("d", 0, _lib.ERR_INVALID_ARG),
    ("N", -1, _lib.ERR_INVALID_ARG),
    ("dtype", 7, _lib.ERR_INVALID_ARG),
    ("tau", float("nan"), _lib.ERR_INVALID_ARG),
    ("tau", 0.0, _lib.ERR_INVALID_ARG),
])
def test_bad_problem_rejected_before_launch(lib, field, value, status):
    p = _lib.Problem(1, 2, 256, 64, 0.125, _lib.BF16, 0)
    setattr(p, field, value)
    assert call_bob(lib, p) == status
    assert lib.fbob_last_error().decode()


def test_null_and_misaligned_pointers_rejected(lib):
    p = _lib.Problem(1, 1, 256, 64, 0.125, _lib.BF16, 0)
    ptrs = [0x1000 * (k + 1) for k in range(14)]
    ptrs[3] = 0
    assert call_bob(lib, p, ptrs) == _lib.ERR_INVALID_ARG
    assert "O" in lib.fbob_last_error().decode()
    ptrs[3] = 0x4008
    assert call_bob(lib, p, ptrs) == _lib.ERR_INVALID_ARG
    assert "aligned" in lib.fbob_last_error().decode()


def test_workspace_checks(lib):
    p = _lib.Problem(1, 1, 256, 64, 0.125, _lib.BF16, 0)
    assert call_bob(lib, p, ws=0) == _lib.ERR_WORKSPACE
    assert call_bob(lib, p, ws_bytes=100) == _lib.ERR_WORKSPACE
    assert call_bob(lib, p, ws=0x10004) == _lib.ERR_WORKSPACE


def test_empty_problem_is_a_noop(lib):
    for B, N in ((0, 256), (1, 0)):
        p = _lib.Problem(B, 4, N, 64, 0.125, _lib.BF16, 0)
        assert call_bob(lib, p, ptrs=[0] * 14, ws=0) == _lib.OK
        assert lib.fbob_attn_fwd(ctypes.byref(p), *[None] * 5, None) == _lib.OK


def test_causal_passes_validation(lib):
    # validation passes for both dtypes; without a GPU the first CUDA call then fails cleanly
    for dt in (_lib.BF16, _lib.FP32):
        p = _lib.Problem(1, 1, 256, 64, 0.125, dt, 1)
        assert call_bob(lib, p) in (_lib.OK, _lib.ERR_CUDA)


def test_ragged_n_passes_validation(lib):
    # any N >= 1 for both dtypes; without a GPU the first CUDA call then fails cleanly
    for dt in (_lib.BF16, _lib.FP32):
        for N in (1, 200, 129):
            p = _lib.Problem(1, 1, N, 64, 0.125, dt, 0)
            assert call_bob(lib, p) in (_lib.OK, _lib.ERR_CUDA)


def test_wait_limit_roundtrip(lib):
    old = lib.fbob_set_wait_limit_ns(12345)
    assert lib.fbob_set_wait_limit_ns(0) == 12345
    assert lib.fbob_set_wait_limit_ns(old) == 2_000_000_000


def test_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()


def test_profile_report_empty_and_toggles(lib):
    assert lib.fbob_profile_enable(0) in (0, 1)
    n = lib.fbob_profile_report(None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    assert lib.fbob_profile_report(buf, n + 1) == n
    assert buf.value.decode() == "{}"
    assert lib.fbob_profile_enable(1) == 0
    assert lib.fbob_profile_enable(0) == 1


def test_stall_hook_toggles_and_defaults_off(lib):
    assert lib.fbob_debug_stall_producer(1) == 0
    assert lib.fbob_debug_stall_producer(0) == 1


def test_four_pass_validates_like_two_pass_and_refuses_fp32(lib):
    """The ablation entry point checks its arguments before any launch, like
    fbob_attn_bob, and runs bf16 inputs only."""
    ptrs = [fake(0x1000 * (k + 1)) for k in range(14)]

    def call(p, ws_bytes=None):
        nb = lib.fbob_bob_workspace_bytes(ctypes.byref(p)) if ws_bytes is None else ws_bytes
        return lib.fbob_attn_bob_four_pass(ctypes.byref(p), *ptrs, fake(0x10000), ctypes.c_size_t(nb), None)

    assert call(_lib.Problem(1, 1, 256, 64, 0.125, _lib.FP32, 0)) == _lib.ERR_UNSUPPORTED
    assert "bf16" in lib.fbob_last_error().decode()
    assert call(_lib.Problem(1, 1, 256, 48, 0.125, _lib.BF16, 0)) == _lib.ERR_UNSUPPORTED
    assert call(_lib.Problem(1, 1, 256, 64, 0.125, _lib.BF16, 0), ws_bytes=8) == _lib.ERR_WORKSPACE
    assert call(_lib.Problem(1, 0, 256, 64, 0.125, _lib.BF16, 0)) == _lib.OK
