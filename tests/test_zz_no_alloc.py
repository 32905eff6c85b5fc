"""GPU test of fbob_attn_bob_noalloc, the BoB entry point whose (alpha, E)
workspace is a fixed device array inside the library.

It exists for callers that cannot hand the library an extra device buffer:
hosts that pass only their own input and output tensors, or loops that must
not call cudaMalloc/cudaFree because those calls can synchronise the device.

Named so that pytest collects it after every other test file.  Through the C
ABI it checks that two calls in a row give the same outputs as fbob_attn_bob
(which takes a caller workspace), that a call allocates no device memory, and
that a problem larger than the fixed workspace is refused before any launch.
Both entry points run the same deterministic kernels on the same inputs and
differ only in where (alpha, E) live, so their outputs must be bit-identical
(which is within every parity tolerance of the other GPU tests); any mix-up of
the workspace would show as a difference.  The cases cover the tensor-core path
(whole and ragged last tiles - the ragged tile reads (alpha, E) back through a
bounds-checked path instead of a bulk copy - and the causal mask) and the fp32
path.
"""

import ctypes
import gc

import numpy as np
import pytest
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
from exact_second_order_attn_gb300 import _lib
from exact_second_order_attn_gb300.build import build
from gpu_helpers import rel_err

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, w, x, O, L, D, outs, causal):
    p = _lib.problem_for(x["Q"], w.tau, causal)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fbob_attn_bob_noalloc(ctypes.byref(p), _vp(x["Q"]), _vp(x["K"]), _vp(x["V"]), _vp(O),
                                     _vp(x["dO"]), _vp(L), _vp(D), _vp(x["UQ"]), _vp(x["UK"]), _vp(x["UV"]),
                                     *[_vp(t) for t in outs], stream)


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (1, 2, 512, 128, "bf16", False),
    (2, 2, 256, 64, "bf16", False),
    (1, 2, 200, 128, "bf16", False),     # ragged last tile
    (2, 1, 333, 64, "bf16", False),      # ragged, N not a multiple of 4
    (1, 2, 384, 128, "bf16", True),      # causal
    (1, 1, 300, 64, "bf16", True),       # causal and ragged
    (1, 1, 200, 64, "fp32", False),
])
def test_two_calls_match_the_workspace_entry_point(lib, B, H, N, d, dtype, causal):
    for seed in (11, 12):   # two calls in a row, different inputs
        w = attn_inputs.small(B, H, N, d, dtype, seed=seed)
        x = {k: v.cuda() for k, v in attn_inputs.make_inputs(w).items()}
        O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, causal=causal)
        first_bwd = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, causal=causal)
        D = first_bwd[3]
        ref = fb.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau,
                          causal=causal)[:4]
        outs = [torch.full_like(O, float("nan")) for _ in range(4)]
        gc.collect()              # tensors left in reference cycles by earlier tests
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        allocated = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(lib, w, x, O, L, D, outs, causal) == _lib.OK, lib.fbob_last_error().decode()
        fb.device_status()
        free_after = torch.cuda.mem_get_info()[0]
        assert torch.cuda.max_memory_allocated() == allocated   # nothing allocated in between
        if seed == 12:   # the first call on the device may load the module
            assert free_before - free_after < (1 << 20)
        for name, a, r in zip(("gQ", "gK", "gV", "gdO"), outs, ref):
            a, r = a.cpu().numpy(), r.cpu().numpy()
            assert np.isfinite(a).all(), name
            assert np.array_equal(a, r), (name, rel_err(a, r))


def test_oversized_problem_is_refused_before_launch(lib):
    rows = (1 << 21) + 128
    p = _lib.Problem(1, 1, rows, 64, 0.125, _lib.BF16, 0)
    fake = [ctypes.c_void_p(0x1000 * (k + 1)) for k in range(14)]
    assert lib.fbob_attn_bob_noalloc(ctypes.byref(p), *fake, None) == _lib.ERR_UNSUPPORTED
    assert "fixed workspace" in lib.fbob_last_error().decode()
