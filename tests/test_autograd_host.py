"""Host test of the autograd wiring (no GPU).

``exact_second_order_attn_gb300.autograd`` only moves tensors between
torch.autograd and the binding.  Here the binding's three calls are replaced
by the fp64 oracle, so gradients and Hessian-vector products taken through
``attention`` must equal PyTorch's own first and second derivatives of a
plain softmax attention written in torch ops.  A wrong cotangent-to-argument
mapping, a dropped dO gradient or a gradient leaking into the saved O / L
would all show up here.
"""

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_second_order_attn_gb300 import _lib
from exact_second_order_attn_gb300 import autograd as ag


def _t(a, like):
    return torch.as_tensor(np.asarray(a), dtype=torch.float64, device=like.device)


@pytest.fixture
def oracle_backend(monkeypatch):
    calls = []

    def fwd(Q, K, V, tau, causal=False, **_):
        calls.append("fwd")
        O, L = orc.attn_fwd(Q.detach().numpy(), K.detach().numpy(), V.detach().numpy(), tau, causal=causal)
        return _t(O, Q), _t(L, Q)

    def bwd(Q, K, V, O, dO, L, tau, causal=False, **_):
        calls.append("bwd")
        dQ, dK, dV, D = orc.attn_bwd(*(x.detach().numpy() for x in (Q, K, V, dO)), tau, causal=causal)
        return _t(dQ, Q), _t(dK, Q), _t(dV, Q), _t(D, Q)

    def bob(Q, K, V, O, dO, L, D, UQ, UK, UV, tau, causal=False, **_):
        calls.append("bob")
        g = orc.attn_bob(*(x.detach().numpy() for x in (Q, K, V, dO, UQ, UK, UV)), tau, causal=causal)
        return tuple(_t(a, Q) for a in g) + (None,)

    monkeypatch.setattr(_lib, "fbob_attn_fwd", fwd)
    monkeypatch.setattr(_lib, "fbob_attn_bwd", bwd)
    monkeypatch.setattr(_lib, "fbob_attn_bob", bob)
    return calls


def torch_attention(Q, K, V, tau, causal=False):
    S = tau * Q @ K.transpose(-1, -2)
    if causal:
        n = S.shape[-1]
        S = S.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), diagonal=1), float("-inf"))
    return torch.softmax(S, dim=-1) @ V


@pytest.mark.parametrize("shape,causal", [((1, 2, 12, 4), False), ((2, 1, 7, 3), False), ((1, 2, 10, 4), True)])
def test_gradients_and_hvp_match_torch_double_backward(oracle_backend, shape, causal):
    g = torch.Generator().manual_seed(5)
    Q, K, V, W, vQ, vK, vV = (torch.randn(shape, generator=g, dtype=torch.float64) for _ in range(7))
    tau = 0.6

    def loss(f):
        return lambda q, k, v: (torch.sin(f(q, k, v, tau, causal)) * W).sum()   # a nonlinear head on O

    x = [t.clone().requires_grad_(True) for t in (Q, K, V)]
    g_ours = torch.autograd.grad(loss(ag.attention)(*x), x)
    x_ref = [t.clone().requires_grad_(True) for t in (Q, K, V)]
    g_ref = torch.autograd.grad(loss(torch_attention)(*x_ref), x_ref)
    for a, b in zip(g_ours, g_ref):
        torch.testing.assert_close(a, b, rtol=1e-10, atol=1e-12)

    hv = ag.hvp(loss(ag.attention), [Q, K, V], [vQ, vK, vV])
    hv_ref = ag.hvp(loss(torch_attention), [Q, K, V], [vQ, vK, vV])
    for a, b in zip(hv, hv_ref):
        torch.testing.assert_close(a, b, rtol=1e-9, atol=1e-11)
    assert oracle_backend.count("bob") == 1   # one BoB call per Hessian-vector product


def test_cotangents_of_unused_gradients_are_zero(oracle_backend):
    g = torch.Generator().manual_seed(6)
    Q, K, V = (torch.randn(1, 1, 9, 4, generator=g, dtype=torch.float64, requires_grad=True) for _ in range(3))
    dQ, dK, dV = torch.autograd.grad(ag.attention(Q, K, V, 0.5).sum(), (Q, K, V), create_graph=True)
    (gQ,) = torch.autograd.grad((dV ** 2).sum(), (Q,))    # only dV used: UQ = UK = 0 reach BoB
    Qr, Kr, Vr = (t.detach().clone().requires_grad_(True) for t in (Q, K, V))
    _, _, dVr = torch.autograd.grad(torch_attention(Qr, Kr, Vr, 0.5).sum(), (Qr, Kr, Vr), create_graph=True)
    (gQr,) = torch.autograd.grad((dVr ** 2).sum(), (Qr,))
    torch.testing.assert_close(gQ, gQr, rtol=1e-9, atol=1e-11)


def test_attention_rejects_non_contiguous_inputs():
    x = torch.zeros(1, 1, 8, 4).transpose(-1, -2)
    with pytest.raises(ValueError, match="contiguous"):
        ag.attention(x, x, x, 1.0)
