"""GPU test of the autograd integration: a Hessian-vector product taken by
double backward through ``exact_second_order_attn_gb300.attention`` runs the
library's BoB kernels and must match the fp64 oracle.

For the loss l = <W, O> the gradient is the first backward with dO = W, and
the Hessian-vector product in direction v = (vQ, vK, vV) is that backward's
vector-Jacobian product with cotangents v: BoB with UQ, UK, UV = vQ, vK, vV.
W and v are drawn at the input precision, so the rounding the autograd layer
applies to them is exact and the oracle sees the same numbers.
"""

import numpy as np
import pytest
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
import oracle.attention as orc
from exact_second_order_attn_gb300.build import build
from gpu_helpers import rel_err

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp32": 2e-5}   # the parity tests' bars


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("B,H,N,d,dtype", [(1, 2, 256, 64, "bf16"), (1, 1, 384, 128, "bf16"), (1, 1, 200, 64, "fp32")])
def test_hvp_through_attention_is_bob(B, H, N, d, dtype):
    w = attn_inputs.small(B, H, N, d, dtype, seed=21)
    x = attn_inputs.make_inputs(w)     # Q, K, V, dO (= W), UQ, UK, UV (= v) at the input dtype
    Q, K, V, W, vQ, vK, vV = (x[k].cuda() for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV"))

    def loss(q, k, v):
        return (fb.attention(q, k, v, w.tau) * W.float()).sum()

    params = [t.clone().requires_grad_(True) for t in (Q, K, V)]
    grads = torch.autograd.grad(loss(*params), params)
    hv = fb.hvp(loss, [Q, K, V], [vQ, vK, vV])
    fb.device_status()

    o = {k: v.double().numpy() for k, v in x.items()}
    dQ, dK, dV, _ = orc.attn_bwd(o["Q"], o["K"], o["V"], o["dO"], w.tau)
    gQ, gK, gV, _ = orc.attn_bob(o["Q"], o["K"], o["V"], o["dO"], o["UQ"], o["UK"], o["UV"], w.tau)
    for name, got, ref in (("dQ", grads[0], dQ), ("dK", grads[1], dK), ("dV", grads[2], dV),
                           ("HvQ", hv[0], gQ), ("HvK", hv[1], gK), ("HvV", hv[2], gV)):
        a = got.double().cpu().numpy()
        assert np.isfinite(a).all(), name
        # gradients come back at the input dtype: allow its rounding on top of the kernel bar
        tol = TOL[dtype] + (2.0 ** -8 if dtype == "bf16" else 0.0)
        assert rel_err(a, ref) <= tol, (name, rel_err(a, ref))
