"""GB300 (sm_103a) exact attention backward-over-backward.

The compute lives in ``libfbob.so`` (hand-written CUDA behind the C ABI in
``include/fbob.h``); this package is its ctypes binding.  Build the library
with ``exact_second_order_attn_gb300.build.build()``.
"""
from ._lib import (  # noqa: F401
    FUNCTIONS, LIB_PATH, FbobError, Problem, attn_bob, attn_bwd, attn_fwd, bob_workspace_bytes,
    device_status, fbob_abi_version, fbob_attn_bob, fbob_attn_bob_four_pass, fbob_attn_bob_noalloc, fbob_attn_bwd, fbob_attn_fwd,
    fbob_bob_workspace_bytes, fbob_debug_stall_producer, fbob_device_status, fbob_profile_enable,
    fbob_profile_report, fbob_set_wait_limit_ns, load, problem_for,
)
from .autograd import attention, hvp  # noqa: F401
