"""GPU parity of the causal path (query i attends to keys j <= i) against
the fp64 oracle's causal mask: forward, first backward and BoB, bf16 inputs
on the tensor-core kernels (several 128-row blocks, so diagonal, below- and
above-diagonal tiles all occur) and fp32 inputs on the FFMA kernels
(ragged N), compared element by element at the parity tests' bars.
"""

import numpy as np
import pytest

import attn_inputs
import exact_second_order_attn_gb300 as fb
from exact_second_order_attn_gb300.build import build
from gpu_helpers import oracle_chain, oracle_inputs, rel_err, run_chain

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp32": 2e-5}
KEYS = ("O", "L", "dQ", "dK", "dV", "D", "gQ", "gK", "gV", "gdO", "alpha", "E")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (1, 2, 256, 64, "bf16"),
    (1, 1, 384, 128, "bf16"),
    (2, 1, 640, 64, "bf16"),
    (1, 1, 1024, 128, "bf16"),
    (1, 1, 200, 64, "fp32"),
    (1, 2, 37, 128, "fp32"),
])
def test_causal_chain_matches_oracle(B, H, N, d, dtype):
    w = attn_inputs.small(B, H, N, d, dtype, seed=41)
    gpu, inp = run_chain(w, causal=True)
    ref = oracle_chain(oracle_inputs(inp), w.tau, causal=True)
    for k in KEYS:
        assert np.isfinite(gpu[k]).all(), k
        e = rel_err(gpu[k], ref[k])
        assert e <= TOL[dtype], (k, e)


def test_causal_differs_from_full_attention():
    # the mask must reach every kernel: each output changes
    w = attn_inputs.small(1, 1, 256, 64, "bf16", seed=42)
    a, inp = run_chain(w, causal=True)
    b, _ = run_chain(w, inp=inp)
    for k in ("O", "dQ", "dK", "dV", "gQ", "gK", "gV", "gdO"):
        assert rel_err(a[k], b[k]) > 0.05, k


def test_causal_hvp_through_autograd():
    import torch
    import oracle.attention as orc
    w = attn_inputs.small(1, 2, 256, 64, "bf16", seed=43)
    x = attn_inputs.make_inputs(w)
    Q, K, V, W, vQ, vK, vV = (x[k].cuda() for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV"))
    hv = fb.hvp(lambda q, k, v: (fb.attention(q, k, v, w.tau, causal=True) * W.float()).sum(), [Q, K, V], [vQ, vK, vV])
    fb.device_status()
    o = {k: v.double().numpy() for k, v in x.items()}
    ref = orc.attn_bob(o["Q"], o["K"], o["V"], o["dO"], o["UQ"], o["UK"], o["UV"], w.tau, causal=True)
    for got, r in zip(hv, ref[:3]):
        assert rel_err(got.double().cpu().numpy(), r) <= 1e-2 + 2.0 ** -8
