"""GPU parity of the four-pass ablation schedule (``fbob_attn_bob_four_pass``:
alpha sweep, E sweep, direct row-output sweep, column pass).  Its four
outputs and the (alpha, E) workspace it leaves are compared element by
element with the fp64 oracle at the bf16 bar, for full, causal and ragged
problems and all head sizes; it must also agree with the two-pass call.
"""

import numpy as np
import pytest
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
from exact_second_order_attn_gb300.build import build
from gpu_helpers import oracle_inputs, rel_err, to_dev
import oracle.attention as orc

pytestmark = pytest.mark.gpu

BF16_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _bob_both(w, causal):
    inp = attn_inputs.make_inputs(w)
    x = to_dev(inp)
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, causal=causal)
    _, _, _, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, causal=causal)
    args = (x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau)
    four = fb.fbob_attn_bob_four_pass(*args, causal=causal)
    two = fb.fbob_attn_bob(*args, causal=causal)
    fb.device_status()
    cpu = lambda outs: [t.double().cpu().numpy() for t in outs]
    return cpu(four), cpu(two), inp


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 512, 64, False),
    (1, 1, 512, 128, False),
    (1, 2, 384, 64, True),
    (1, 1, 384, 128, True),
    (1, 1, 333, 128, False),
    (2, 1, 200, 64, True),
    (1, 1, 256, 96, False),
    (1, 1, 256, 32, True),
])
def test_four_pass_matches_oracle_and_two_pass(B, H, N, d, causal):
    w = attn_inputs.small(B, H, N, d, "bf16", seed=81)
    four, two, inp = _bob_both(w, causal)
    x = oracle_inputs(inp)
    args = [x[k] for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV")]
    ref = list(orc.attn_bob(*args, w.tau, causal=causal))
    ref += list(orc.bob_row_scalars(*args, w.tau, causal=causal))
    got = four[:4] + [four[4][..., 0], four[4][..., 1]]
    names = ("gQ", "gK", "gV", "gdO", "alpha", "E")
    for k, g, r in zip(names, got, ref):
        assert np.isfinite(g).all(), k
        assert rel_err(g, r) <= BF16_TOL, (k, rel_err(g, r))
    for k, a, b in zip(names[:4], four[:4], two[:4]):
        assert rel_err(a, b) <= BF16_TOL, (k, rel_err(a, b))


def test_four_pass_rejects_fp32():
    w = attn_inputs.small(1, 1, 128, 64, "fp32", seed=82)
    x = to_dev(attn_inputs.make_inputs(w))
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau)
    _, _, _, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau)
    with pytest.raises(fb.FbobError):
        fb.fbob_attn_bob_four_pass(x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau)
    torch.cuda.synchronize()
