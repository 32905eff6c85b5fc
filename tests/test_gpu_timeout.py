"""Failure detection on the GPU without a GPU fault.

Every device-side wait of the tensor-core kernels is bounded.  Here the TMA
producer is told to withhold its first streamed tile (a barrier that nothing
will complete), so the consumers' waits run out: each CTA gives up, drains
what it has in flight, frees its TMEM and returns; the host reads
FBOB_ERR_TIMEOUT from the device status word; and the context stays usable -
the same call afterwards gives the same results as before.
"""

import numpy as np
import pytest
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
from exact_second_order_attn_gb300 import _lib
from exact_second_order_attn_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_withheld_tile_times_out_and_context_survives(d):
    build()
    w = attn_inputs.small(1, 2, 256, d, "bf16", seed=5)
    x = {k: v.cuda() for k, v in attn_inputs.make_inputs(w).items()}
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau)
    _, _, _, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau)
    args = (x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau)
    ref = [t.clone() for t in fb.attn_bob(*args)[:4]]
    fb.device_status()

    old_limit = fb.fbob_set_wait_limit_ns(50_000_000)   # 50 ms per wait
    fb.fbob_debug_stall_producer(True)
    try:
        fb.attn_bob(*args)
        with pytest.raises(fb.FbobError) as err:
            fb.device_status()
        assert err.value.status == _lib.ERR_TIMEOUT
    finally:
        fb.fbob_debug_stall_producer(False)
        fb.fbob_set_wait_limit_ns(old_limit)

    fb.device_status()   # the status word was cleared by the read above
    again = fb.attn_bob(*args)[:4]
    fb.device_status()
    torch.cuda.synchronize()
    for a, r in zip(again, ref):
        np.testing.assert_array_equal(a.cpu().numpy(), r.cpu().numpy())
