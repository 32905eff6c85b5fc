"""ctypes binding of libfbob.so: argument marshalling only.

Each function checks tensor shapes/dtypes/devices, passes raw device pointers
and the current torch CUDA stream to the C ABI (include/fbob.h) and raises
``FbobError`` on a non-OK status.  Every step of the computation runs in the
library's kernels; there is no fallback of any kind - if the library is not
built the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfbob.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
BF16, FP32 = 0, 1

FUNCTIONS = (
    "fbob_attn_fwd", "fbob_attn_bwd", "fbob_bob_workspace_bytes", "fbob_attn_bob",
    "fbob_device_status", "fbob_set_wait_limit_ns", "fbob_status_string", "fbob_last_error",
    "fbob_abi_version", "fbob_attn_bob_noalloc", "fbob_profile_enable", "fbob_profile_report",
    "fbob_debug_stall_producer", "fbob_attn_bob_four_pass",
)


class Problem(ctypes.Structure):
    """fbob_problem: B x H heads of N x d matrices, score scale tau."""
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
                ("tau", ctypes.c_float), ("dtype", ctypes.c_int), ("causal", ctypes.c_int)]


class FbobError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        super().__init__(f"{_status_name(status)}: {detail}")


_lib = None


def load():
    """Load libfbob.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with exact_second_order_attn_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, cp, st = ctypes.c_void_p, ctypes.POINTER(Problem), ctypes.c_int
    lib.fbob_attn_fwd.argtypes = [cp] + [vp] * 6
    lib.fbob_attn_fwd.restype = st
    lib.fbob_attn_bwd.argtypes = [cp] + [vp] * 11
    lib.fbob_attn_bwd.restype = st
    lib.fbob_bob_workspace_bytes.argtypes = [cp]
    lib.fbob_bob_workspace_bytes.restype = ctypes.c_size_t
    lib.fbob_attn_bob.argtypes = [cp] + [vp] * 15 + [ctypes.c_size_t, vp]
    lib.fbob_attn_bob.restype = st
    lib.fbob_attn_bob_four_pass.argtypes = [cp] + [vp] * 15 + [ctypes.c_size_t, vp]
    lib.fbob_attn_bob_four_pass.restype = st
    lib.fbob_attn_bob_noalloc.argtypes = [cp] + [vp] * 15
    lib.fbob_attn_bob_noalloc.restype = st
    lib.fbob_device_status.argtypes = [vp]
    lib.fbob_device_status.restype = st
    lib.fbob_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fbob_set_wait_limit_ns.restype = ctypes.c_ulonglong
    lib.fbob_status_string.argtypes = [st]
    lib.fbob_status_string.restype = ctypes.c_char_p
    lib.fbob_last_error.argtypes = []
    lib.fbob_last_error.restype = ctypes.c_char_p
    lib.fbob_profile_enable.argtypes = [ctypes.c_int]
    lib.fbob_profile_enable.restype = ctypes.c_int
    lib.fbob_profile_report.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
    lib.fbob_profile_report.restype = ctypes.c_int
    lib.fbob_debug_stall_producer.argtypes = [ctypes.c_int]
    lib.fbob_debug_stall_producer.restype = ctypes.c_int
    lib.fbob_abi_version.argtypes = []
    lib.fbob_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def _status_name(s):
    try:
        return load().fbob_status_string(s).decode()
    except Exception:  # library missing while formatting an error
        return f"status {s}"


def _check(status):
    if status != OK:
        raise FbobError(status, load().fbob_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def problem_for(Q: torch.Tensor, tau: float, causal: bool = False) -> Problem:
    if Q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    B, H, N, d = Q.shape
    if Q.dtype == torch.bfloat16:
        dt = BF16
    elif Q.dtype == torch.float32:
        dt = FP32
    else:
        raise TypeError(f"unsupported input dtype {Q.dtype}")
    return Problem(B, H, N, d, float(tau), dt, int(bool(causal)))


def _same(ref, *ts, dtype=None, shape=None):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.device != ref.device:
            raise ValueError("all tensors must be on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"expected {dtype}, got {t.dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _empty(ref, shape=None):
    return torch.empty(ref.shape if shape is None else shape, dtype=torch.float32, device=ref.device)


def fbob_attn_fwd(Q, K, V, tau, O=None, L=None, stream=None, causal=False):
    """(O, L) = forward; allocates O, L if not given.  ``causal``: query i
    attends to keys j <= i."""
    p = problem_for(Q, tau, causal)
    O = _empty(Q) if O is None else O
    L = _empty(Q, Q.shape[:3]) if L is None else L
    _same(Q, K, V, dtype=Q.dtype, shape=Q.shape)
    _same(Q, O, dtype=torch.float32, shape=Q.shape)
    _same(Q, L, dtype=torch.float32, shape=Q.shape[:3])
    _check(load().fbob_attn_fwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), _stream(stream)))
    return O, L


def fbob_attn_bwd(Q, K, V, O, dO, L, tau, dQ=None, dK=None, dV=None, D=None, stream=None, causal=False):
    """(dQ, dK, dV, D) = first backward; allocates outputs if not given."""
    p = problem_for(Q, tau, causal)
    dQ = _empty(Q) if dQ is None else dQ
    dK = _empty(Q) if dK is None else dK
    dV = _empty(Q) if dV is None else dV
    D = _empty(Q, Q.shape[:3]) if D is None else D
    _same(Q, K, V, dO, dtype=Q.dtype, shape=Q.shape)
    _same(Q, O, dQ, dK, dV, dtype=torch.float32, shape=Q.shape)
    _same(Q, L, D, dtype=torch.float32, shape=Q.shape[:3])
    _check(load().fbob_attn_bwd(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L),
                                _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(D), _stream(stream)))
    return dQ, dK, dV, D


def fbob_bob_workspace_bytes(Q):
    p = problem_for(Q, 1.0)
    return int(load().fbob_bob_workspace_bytes(ctypes.byref(p)))


def _bob_call(entry, Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ, gK, gV, gdO, workspace, stream, causal):
    """Marshal the arguments of one of the workspace-taking BoB entry points."""
    p = problem_for(Q, tau, causal)
    gQ = _empty(Q) if gQ is None else gQ
    gK = _empty(Q) if gK is None else gK
    gV = _empty(Q) if gV is None else gV
    gdO = _empty(Q) if gdO is None else gdO
    if workspace is None:
        workspace = _empty(Q, tuple(Q.shape[:3]) + (2,))
    _same(Q, K, V, dO, UQ, UK, UV, dtype=Q.dtype, shape=Q.shape)
    _same(Q, O, gQ, gK, gV, gdO, dtype=torch.float32, shape=Q.shape)
    _same(Q, L, D, dtype=torch.float32, shape=Q.shape[:3])
    _same(Q, workspace, dtype=torch.float32)
    nbytes = workspace.numel() * 4
    _check(getattr(load(), entry)(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(D),
                                  _ptr(UQ), _ptr(UK), _ptr(UV), _ptr(gQ), _ptr(gK), _ptr(gV), _ptr(gdO),
                                  _ptr(workspace), ctypes.c_size_t(nbytes), _stream(stream)))
    return gQ, gK, gV, gdO, workspace


def fbob_attn_bob(Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ=None, gK=None, gV=None, gdO=None,
                  workspace=None, stream=None, causal=False):
    """(gQ, gK, gV, gdO, workspace) = BoB; allocates outputs/workspace if not given.

    ``workspace`` is a float32 tensor [B, H, N, 2] holding (alpha, E) per row.
    """
    return _bob_call("fbob_attn_bob", Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ, gK, gV, gdO, workspace,
                     stream, causal)


def fbob_attn_bob_four_pass(Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ=None, gK=None, gV=None, gdO=None,
                            workspace=None, stream=None, causal=False):
    """BoB on the four-pass schedule (the ablation of the two-pass one; bf16
    only): same arguments and results as :func:`fbob_attn_bob`."""
    return _bob_call("fbob_attn_bob_four_pass", Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ, gK, gV, gdO,
                     workspace, stream, causal)


def fbob_attn_bob_noalloc(Q, K, V, O, dO, L, D, UQ, UK, UV, tau, gQ=None, gK=None, gV=None, gdO=None,
                          stream=None, causal=False):
    """(gQ, gK, gV, gdO) = BoB with the library's fixed workspace (no workspace argument)."""
    p = problem_for(Q, tau, causal)
    gQ = _empty(Q) if gQ is None else gQ
    gK = _empty(Q) if gK is None else gK
    gV = _empty(Q) if gV is None else gV
    gdO = _empty(Q) if gdO is None else gdO
    _same(Q, K, V, dO, UQ, UK, UV, dtype=Q.dtype, shape=Q.shape)
    _same(Q, O, gQ, gK, gV, gdO, dtype=torch.float32, shape=Q.shape)
    _same(Q, L, D, dtype=torch.float32, shape=Q.shape[:3])
    _check(load().fbob_attn_bob_noalloc(ctypes.byref(p), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L),
                                        _ptr(D), _ptr(UQ), _ptr(UK), _ptr(UV), _ptr(gQ), _ptr(gK), _ptr(gV),
                                        _ptr(gdO), _stream(stream)))
    return gQ, gK, gV, gdO


def fbob_device_status(stream=None):
    """Synchronise the stream and raise FbobError if a kernel timed out a wait."""
    _check(load().fbob_device_status(_stream(stream)))


def fbob_set_wait_limit_ns(ns: int) -> int:
    return int(load().fbob_set_wait_limit_ns(ctypes.c_ulonglong(ns)))


def fbob_profile_enable(on: bool) -> bool:
    return bool(load().fbob_profile_enable(int(bool(on))))


def fbob_profile_report() -> dict:
    """Per-kernel {name: (launches, total_ms, min_ms, max_ms)} since the last report."""
    import json
    n = load().fbob_profile_report(None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    load().fbob_profile_report(buf, n + 1)
    return {k: tuple(v) for k, v in json.loads(buf.value.decode()).items()}


def fbob_debug_stall_producer(stall: bool) -> bool:
    return bool(load().fbob_debug_stall_producer(int(bool(stall))))


def fbob_abi_version() -> int:
    return int(load().fbob_abi_version())


# short aliases
attn_fwd = fbob_attn_fwd
attn_bwd = fbob_attn_bwd
attn_bob = fbob_attn_bob
bob_workspace_bytes = fbob_bob_workspace_bytes
device_status = fbob_device_status
