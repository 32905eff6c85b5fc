"""Pins of the oracle's causal mask (CPU only).

The pages do not state a mask; the causal variant is the plain definition
(query i attends to keys j <= i).  It is pinned to torch.autograd through a
torch masked softmax (first and double backward), to brute-force loops, to
the prefix property of causal attention (rows before k see only keys before
k, exactly like non-causal attention on the prefix), to its own unmasked
counterpart at the last row, and to row blocking and row sampling.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as orc


def inputs(rng, N, d, sig=(1,) * 7, H=1):
    return [rng.standard_normal((H, N, d)) * s for s in sig]


def _torch_causal_fwd(Q, K, V, tau):
    N = Q.shape[-2]
    S = tau * Q @ K.transpose(-1, -2)
    mask = torch.triu(torch.ones(N, N, dtype=torch.bool), diagonal=1)
    return torch.softmax(S.masked_fill(mask, float("-inf")), dim=-1) @ V


def test_causal_fwd_bruteforce_loops():
    rng = np.random.default_rng(31)
    N, d, tau = 9, 3, 0.7
    Q, K, V = (x[0] for x in inputs(rng, N, d)[:3])
    O, L = orc.attn_fwd(Q[None], K[None], V[None], tau, causal=True)
    for i in range(N):
        s = [tau * sum(Q[i, c] * K[j, c] for c in range(d)) for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for c in range(d):
            assert abs(O[0, i, c] - sum(e[j] * V[j, c] for j in range(i + 1)) / z) < 1e-12
        assert abs(L[0, i] - (m + math.log(z))) < 1e-12


@pytest.mark.parametrize("N,d", [(24, 8), (37, 5), (1, 4)])
def test_causal_bwd_matches_torch_autograd(N, d):
    rng = np.random.default_rng(32)
    Q, K, V, dO = inputs(rng, N, d)[:4]
    tau = 0.45
    dQ, dK, dV, D = orc.attn_bwd(Q, K, V, dO, tau, causal=True)
    tQ, tK, tV = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    O = _torch_causal_fwd(tQ, tK, tV, tau)
    gq, gk, gv = torch.autograd.grad(O, (tQ, tK, tV), torch.tensor(dO))
    for a, b in ((dQ, gq), (dK, gk), (dV, gv)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(D, (dO * O.detach().numpy()).sum(-1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("N,d,H,sig", [
    (16, 8, 1, (1,) * 7),
    (37, 5, 2, (1,) * 7),
    (64, 16, 1, (4, 4, 1, 1, 1, 1, 1)),
    (1, 3, 1, (1,) * 7),
])
def test_causal_bob_matches_torch_double_backward(N, d, H, sig):
    rng = np.random.default_rng(33)
    X = inputs(rng, N, d, sig, H)
    tau = 1.0 / math.sqrt(d)
    ours = orc.attn_bob(*X, tau, causal=True)
    tQ, tK, tV, tdO = (torch.tensor(x, requires_grad=True) for x in X[:4])
    O = _torch_causal_fwd(tQ, tK, tV, tau)
    dQ, dK, dV = torch.autograd.grad(O, (tQ, tK, tV), tdO, create_graph=True)
    f = sum((g * torch.tensor(u)).sum() for g, u in zip((dQ, dK, dV), X[4:]))
    ref = [g.numpy() for g in torch.autograd.grad(f, (tQ, tK, tV, tdO))]
    for a, b in zip(ours, ref):
        assert np.abs(a - b).max() <= 1e-11 * max(1e-30, np.abs(b).max()) + 1e-14


def test_prefix_rows_equal_noncausal_attention_on_the_prefix():
    rng = np.random.default_rng(34)
    N, k, d, tau = 30, 11, 6, 0.5
    Q, K, V, dO, UQ, UK, UV = inputs(rng, N, d)
    O, L = orc.attn_fwd(Q, K, V, tau, causal=True)
    Op, Lp = orc.attn_fwd(Q[:, :k], K[:, :k], V[:, :k], tau, causal=True)
    np.testing.assert_allclose(O[:, :k], Op, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L[:, :k], Lp, rtol=1e-12, atol=1e-13)
    # the last row of causal attention is the unmasked row
    Of, _ = orc.attn_fwd(Q, K, V, tau)
    np.testing.assert_allclose(O[:, -1], Of[:, -1], rtol=1e-12, atol=1e-13)
    # keys after k receive nothing from the first k rows: zero their queries' cotangents
    # and dO beyond k, then dK, dV of keys >= k vanish
    dOz = dO.copy()
    dOz[:, k:] = 0
    _, dK, dV, _ = orc.attn_bwd(Q, K, V, dOz, tau, causal=True)
    assert np.abs(dK[:, k:]).max() < 1e-14 and np.abs(dV[:, k:]).max() < 1e-14


def test_causal_row_blocking_and_sampling(monkeypatch):
    rng = np.random.default_rng(35)
    N, d, tau = 50, 6, 0.5
    X = inputs(rng, N, d, H=2)
    full = orc.attn_bob(*X, tau, causal=True)
    alpha, E = orc.bob_row_scalars(*X, tau, causal=True)
    rows = [0, 7, 49]
    sq, so = orc.bob_sampled_rows(*(x[1] for x in X), tau, rows, causal=True)
    np.testing.assert_allclose(sq, full[0][1][rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(so, full[3][1][rows], rtol=1e-12, atol=1e-13)
    _, dK, dV, _ = orc.attn_bwd(*X[:4], tau, causal=True)
    cols = [0, 7, 48, 49]
    got = orc.bob_sampled_cols(*(x[1] for x in X), tau, cols, causal=True)
    for g, ref in zip(got, (dK[1], dV[1], full[1][1], full[2][1])):
        np.testing.assert_allclose(g, ref[cols], rtol=1e-12, atol=1e-13)
    monkeypatch.setattr(orc, "_BLOCK_ELEMS", 4 * N)      # 4-row blocks, ragged tail
    blocked = orc.attn_bob(*X, tau, causal=True)
    for a, b in zip(full, blocked):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    ab, Eb = orc.bob_row_scalars(*X, tau, causal=True)
    np.testing.assert_allclose(alpha, ab, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(E, Eb, rtol=1e-12, atol=1e-13)


def test_mask_changes_the_result():
    # guard against a mask that silently does nothing
    rng = np.random.default_rng(36)
    X = inputs(rng, 12, 4)
    a = orc.attn_bob(*X, 0.5, causal=True)
    b = orc.attn_bob(*X, 0.5)
    assert np.abs(a[0] - b[0]).max() > 1e-3
