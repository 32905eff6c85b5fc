"""Pins of the oracle's four-pass restatement (``bob_four_pass_rows``), the
schedule the affine structure collapses to two (evolve.pub review,
Strengths).  Its outputs must be the exact BoB - checked against torch's own
fp64 double backward, not against the oracle's two-pass code - and its
scalars must relate to the two-pass ones as the reading states: the same
alpha, and En = E - 2 alpha D.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as orc


def _torch_bob(Q, K, V, dO, UQ, UK, UV, tau, causal):
    tQ, tK, tV, tdO = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, dO))
    S = tau * tQ @ tK.transpose(-1, -2)
    if causal:
        n = S.shape[-1]
        S = S.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    O = torch.softmax(S, dim=-1) @ tV
    dQ, dK, dV = torch.autograd.grad(O, (tQ, tK, tV), tdO, create_graph=True)
    f = (dQ * torch.tensor(UQ)).sum() + (dK * torch.tensor(UK)).sum() + (dV * torch.tensor(UV)).sum()
    return [g.numpy() for g in torch.autograd.grad(f, (tQ, tK, tV, tdO))]


@pytest.mark.parametrize("N,d,H,causal", [(24, 8, 1, False), (37, 5, 2, False), (30, 6, 2, True), (1, 4, 1, False)])
def test_four_pass_outputs_match_torch_double_backward(N, d, H, causal):
    rng = np.random.default_rng(71)
    X = [rng.standard_normal((H, N, d)) for _ in range(7)]
    tau = 1.0 / math.sqrt(d)
    ours = orc.attn_bob_four_pass(*X, tau, causal=causal)[:4]
    ref = _torch_bob(*X, tau, causal)
    for a, b in zip(ours, ref):
        scale = max(1e-30, np.abs(b).max())
        assert np.abs(a - b).max() <= 1e-11 * scale + 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_four_pass_scalars_relate_to_the_two_pass_ones(causal):
    rng = np.random.default_rng(72)
    N, d, tau = 33, 7, 0.4
    X = [rng.standard_normal((2, N, d)) for _ in range(7)]
    *_, alpha4, En = orc.attn_bob_four_pass(*X, tau, causal=causal)
    alpha, E = orc.bob_row_scalars(*X, tau, causal=causal)
    D = orc.attn_bwd(X[0], X[1], X[2], X[3], tau, causal=causal)[3]
    np.testing.assert_allclose(alpha4, alpha, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(En, E - 2 * alpha * D, rtol=1e-11, atol=1e-12)


def test_dropping_the_alpha_term_of_pbar_breaks_the_result():
    """The alpha dP term of Pbar is what makes the natural E need a second
    pass; without it the outputs are wrong (a planted mistake in a copy of
    the restatement must be caught by the torch pin)."""
    rng = np.random.default_rng(73)
    N, d, tau = 20, 6, 0.5
    Q, K, V, dO, UQ, UK, UV = (rng.standard_normal((N, d)) for _ in range(7))
    P = torch.softmax(torch.tensor(tau * Q @ K.T), dim=-1).numpy()
    O, dP = P @ V, dO @ V.T
    D = (dO * O).sum(1)[:, None]
    B, C = tau * (UQ @ K.T + Q @ UK.T), dO @ UV.T
    P_bar_wrong = C + B * (dP - D)                 # alpha dP dropped
    S_bar = P * (P_bar_wrong - (P * P_bar_wrong).sum(1, keepdims=True))
    dS = P * (dP - D)
    gQ_wrong = tau * (dS @ UK + S_bar @ K)
    gQ_ref = _torch_bob(Q[None], K[None], V[None], dO[None], UQ[None], UK[None], UV[None], tau, False)[0][0]
    gQ_ours = orc.bob_four_pass_rows(Q, K, V, dO, UQ, UK, UV, tau)[0]
    assert np.abs(gQ_wrong - gQ_ref).max() > 1e-3 * np.abs(gQ_ref).max()
    np.testing.assert_allclose(gQ_ours, gQ_ref, rtol=1e-10, atol=1e-12)
