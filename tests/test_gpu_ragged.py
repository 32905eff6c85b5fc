"""GPU parity for N that is not a multiple of the 128-row block on the
tensor-core (bf16) kernels, with and without the causal mask: the last row
block is partly past the end and the last streamed tile crosses N, so the
zero-filled TMA rows, the column mask at N, the guarded row loads and stores
and the bounds-checked per-tile vectors are all exercised.  All twelve
outputs are compared element by element with the fp64 oracle at the bf16 bar.
"""

import numpy as np
import pytest

import attn_inputs
from exact_second_order_attn_gb300.build import build
from gpu_helpers import oracle_chain, oracle_inputs, rel_err, run_chain

pytestmark = pytest.mark.gpu

BF16_TOL = 1e-2
KEYS = ("O", "L", "dQ", "dK", "dV", "D", "gQ", "gK", "gV", "gdO", "alpha", "E")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 200, 64, False),     # one partial block, last 64-row tile partly valid
    (1, 1, 129, 128, False),    # one row past a block boundary
    (2, 1, 333, 64, False),
    (1, 1, 1000, 128, False),
    (1, 1, 1, 64, False),       # a single row
    (1, 2, 300, 64, True),
    (1, 1, 450, 128, True),
])
def test_ragged_chain_matches_oracle(B, H, N, d, causal):
    w = attn_inputs.small(B, H, N, d, "bf16", seed=51)
    gpu, inp = run_chain(w, causal=causal)
    ref = oracle_chain(oracle_inputs(inp), w.tau, causal=causal)
    for k in KEYS:
        assert np.isfinite(gpu[k]).all(), k
        e = rel_err(gpu[k], ref[k])
        assert e <= BF16_TOL, (k, e)
