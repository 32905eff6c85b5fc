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


def _rnd(a, dtype):
    """Round an fp64 array to the input dtype the way the autograd layer does
    (a torch cast), back in fp64."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).double().numpy()


@pytest.mark.parametrize("B,H,N,d,dtype,sigma", [
    (1, 2, 256, 64, "bf16", (1.0,) * 7),
    (1, 1, 384, 128, "bf16", (1.0,) * 7),
    (1, 1, 200, 64, "fp32", (1.0,) * 7),
    (8, 12, 1024, 64, "bf16", (1.0, 1.0, 1.0, 0.1, 0.1, 0.1, 0.1)),   # the GPT-2-Small shape
])
def test_hvp_of_a_loss_nonlinear_in_o(B, H, N, d, dtype, sigma):
    """l = 1/2 <W, O o O>: the gradient's incoming dO = W o O depends on the
    parameters, so the Hessian-vector product has a second term through dO.
    With (gQ, gK, gV, gdO) = BoB at dO = W o O with cotangents v, it is
        H v = (gQ, gK, gV) + first backward with dO' = W o gdO,
    the chain rule through dO = W o O(Q, K, V).  The oracle mirrors the
    autograd layer's roundings to the input dtype (dO, gdO and dO')."""
    w = attn_inputs.small(B, H, N, d, dtype, sigma=sigma, seed=23)
    x = attn_inputs.make_inputs(w)     # Q, K, V, W (in dO), v (in UQ, UK, UV) at the input dtype
    Q, K, V, W, vQ, vK, vV = (x[k].cuda() for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV"))

    def loss(q, k, v):
        o = fb.attention(q, k, v, w.tau)
        return 0.5 * (o * o * W.float()).sum()

    params = [t.clone().requires_grad_(True) for t in (Q, K, V)]
    grads = torch.autograd.grad(loss(*params), params)
    hv = fb.hvp(loss, [Q, K, V], [vQ, vK, vV])
    fb.device_status()

    heads = [(b, h) for b in range(B) for h in range(H)]
    if len(heads) > 4:
        heads = [heads[0], heads[len(heads) // 3], heads[2 * len(heads) // 3], heads[-1]]
    for b, h in heads:
        o = {k: v[b, h].double().numpy() for k, v in x.items()}
        Wd = o["dO"]
        O, _ = orc.attn_fwd_head(o["Q"], o["K"], o["V"], w.tau)
        dO = _rnd(Wd * O, dtype)
        dQ, dK, dV, _ = orc.attn_bwd(o["Q"][None], o["K"][None], o["V"][None], dO[None], w.tau)
        gQ, gK, gV, gdO = orc.attn_bob(o["Q"][None], o["K"][None], o["V"][None], dO[None],
                                       o["UQ"][None], o["UK"][None], o["UV"][None], w.tau)
        dO2 = _rnd(Wd * _rnd(gdO[0], dtype), dtype)
        hQ, hK, hV, _ = orc.attn_bwd(o["Q"][None], o["K"][None], o["V"][None], dO2[None], w.tau)
        ref = {"dQ": dQ[0], "dK": dK[0], "dV": dV[0],
               "HvQ": gQ[0] + hQ[0], "HvK": gK[0] + hK[0], "HvV": gV[0] + hV[0]}
        got = {"dQ": grads[0], "dK": grads[1], "dV": grads[2], "HvQ": hv[0], "HvK": hv[1], "HvV": hv[2]}
        for name, r in ref.items():
            a = got[name][b, h].double().cpu().numpy()
            assert np.isfinite(a).all(), name
            # the kernel bar, plus the returned gradient's rounding to the input dtype and,
            # for H v, the bf16 sum of its two terms
            tol = TOL[dtype] + (2.0 ** -7 if dtype == "bf16" else 0.0)
            assert rel_err(a, r) <= tol, (name, (b, h), rel_err(a, r))
