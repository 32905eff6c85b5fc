"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against an independent fact: a library routine,
brute-force loops, torch.autograd, a sympy symbolic derivative, central finite
differences, the closed-form reduction printed on the pages, a hand-computed
fixture, or an exact invariant of the mathematics.  Together they are chosen
so that a dropped term, a wrong sign or index, or a transposed operand anywhere
in the oracle fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle.attention as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def inputs(rng, N, d, sig=(1,) * 7, H=1):
    return [rand(rng, H, N, d, scale=s) for s in sig]


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def test_fwd_matches_scipy_softmax_logsumexp():
    rng = np.random.default_rng(1)
    Q, K, V = (rand(rng, 2, 40, 16) for _ in range(3))
    tau = 0.3
    O, L = orc.attn_fwd(Q, K, V, tau)
    S = tau * np.einsum("hid,hjd->hij", Q, K)
    P = scipy.special.softmax(S, axis=-1)
    np.testing.assert_allclose(O, P @ V, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(L, scipy.special.logsumexp(S, axis=-1), rtol=1e-13, atol=1e-13)


def test_fwd_bruteforce_loops():
    rng = np.random.default_rng(2)
    N, d, tau = 3, 2, 0.7
    Q, K, V = (rand(rng, N, d) for _ in range(3))
    O, L = orc.attn_fwd_head(Q, K, V, tau)
    for i in range(N):
        s = [tau * sum(Q[i, c] * K[j, c] for c in range(d)) for j in range(N)]
        z = sum(math.exp(x) for x in s)
        assert abs(L[i] - math.log(z)) < 1e-13
        for c in range(d):
            o = sum(math.exp(s[j]) / z * V[j, c] for j in range(N))
            assert abs(O[i, c] - o) < 1e-13


def test_fwd_golden_hand_values():
    with open(os.path.join(GOLDEN, "lemma_e2_hand.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        Q, K, W = (np.array(case[k]) for k in ("Q", "K", "W"))
        O, L = orc.attn_fwd_head(Q, K, W, case["tau"])
        np.testing.assert_allclose(O, case["expected_O_with_V_eq_W"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(L, case["expected_L"], rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# first backward
# ---------------------------------------------------------------------------

def _torch_fwd(Q, K, V, tau):
    return torch.softmax(tau * Q @ K.transpose(-1, -2), dim=-1) @ V


@pytest.mark.parametrize("N,d", [(24, 8), (37, 5), (1, 4)])
def test_bwd_matches_torch_autograd(N, d):
    rng = np.random.default_rng(3)
    Q, K, V, dO = inputs(rng, N, d)[:4]
    tau = 0.45
    dQ, dK, dV, D = orc.attn_bwd(Q, K, V, dO, tau)
    tQ, tK, tV = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    O = _torch_fwd(tQ, tK, tV, tau)
    gq, gk, gv = torch.autograd.grad(O, (tQ, tK, tV), torch.tensor(dO))
    for a, b in ((dQ, gq), (dK, gk), (dV, gv)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(D, (dO * O.detach().numpy()).sum(-1), rtol=1e-12, atol=1e-12)


def test_bwd_central_differences_of_forward():
    rng = np.random.default_rng(4)
    N, d, tau = 12, 6, 0.5
    Q, K, V, dO = inputs(rng, N, d)[:4]
    vQ, vK, vV = (rand(rng, 1, N, d) for _ in range(3))
    dQ, dK, dV, _ = orc.attn_bwd(Q, K, V, dO, tau)
    h = 1e-5

    def loss(s):
        O, _ = orc.attn_fwd(Q + s * vQ, K + s * vK, V + s * vV, tau)
        return float((dO * O).sum())

    fd = (loss(h) - loss(-h)) / (2 * h)
    an = float((dQ * vQ).sum() + (dK * vK).sum() + (dV * vV).sum())
    assert abs(fd - an) <= 1e-8 * max(1.0, abs(an))


# ---------------------------------------------------------------------------
# backward over backward
# ---------------------------------------------------------------------------

def _torch_bob(Q, K, V, dO, UQ, UK, UV, tau):
    tQ, tK, tV, tdO = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, dO))
    O = _torch_fwd(tQ, tK, tV, tau)
    dQ, dK, dV = torch.autograd.grad(O, (tQ, tK, tV), tdO, create_graph=True)
    f = (dQ * torch.tensor(UQ)).sum() + (dK * torch.tensor(UK)).sum() + (dV * torch.tensor(UV)).sum()
    return [g.numpy() for g in torch.autograd.grad(f, (tQ, tK, tV, tdO))]


@pytest.mark.parametrize("N,d,H,sig", [
    (16, 8, 1, (1,) * 7),
    (37, 5, 2, (1,) * 7),                       # ragged, several heads
    (64, 16, 1, (4, 4, 1, 1, 1, 1, 1)),         # peaky rows
    (48, 8, 1, (1, 1, 1, .1, .1, .1, .1)),      # small cotangents
    (1, 3, 1, (1,) * 7),                        # one key: softmax is constant
])
def test_bob_matches_torch_double_backward(N, d, H, sig):
    rng = np.random.default_rng(5)
    X = inputs(rng, N, d, sig, H)
    tau = 1.0 / math.sqrt(d)
    ours = orc.attn_bob(*X, tau)
    ref = _torch_bob(*X, tau)
    for a, b in zip(ours, ref):
        scale = max(1e-30, np.abs(b).max())
        assert np.abs(a - b).max() <= 1e-11 * scale + 1e-14


def test_bob_adjoint_identity_central_differences():
    """<J_g^T U, v> = <U, J_g v>, with J_g v from central differences of the
    oracle's own fp64 first backward (N = 16, d = 8)."""
    rng = np.random.default_rng(6)
    N, d, tau = 16, 8, 1.0 / math.sqrt(8)
    Q, K, V, dO, UQ, UK, UV = inputs(rng, N, d)
    v = [rand(rng, 1, N, d) for _ in range(4)]
    gQ, gK, gV, gdO = orc.attn_bob(Q, K, V, dO, UQ, UK, UV, tau)
    h = 1e-5
    plus = orc.attn_bwd(Q + h * v[0], K + h * v[1], V + h * v[2], dO + h * v[3], tau)
    minus = orc.attn_bwd(Q - h * v[0], K - h * v[1], V - h * v[2], dO - h * v[3], tau)
    jv = [(p - m) / (2 * h) for p, m in zip(plus[:3], minus[:3])]
    rhs = float((UQ * jv[0]).sum() + (UK * jv[1]).sum() + (UV * jv[2]).sum())
    lhs = float((gQ * v[0]).sum() + (gK * v[1]).sum() + (gV * v[2]).sum() + (gdO * v[3]).sum())
    assert abs(lhs - rhs) <= 1e-8 * max(1.0, abs(rhs))


def test_bob_sympy_symbolic_second_derivative():
    """Differentiate the scalar <dO, O> twice symbolically (N = 2, d = 2)."""
    sp = pytest.importorskip("sympy")
    N, d, tau = 2, 2, sp.Rational(3, 5)
    sym = {n: sp.Matrix(N, d, lambda i, c: sp.Symbol(f"{n}{i}{c}")) for n in ("Q", "K", "V", "G")}
    Q, K, V, G = sym["Q"], sym["K"], sym["V"], sym["G"]
    loss = 0
    for i in range(N):
        s = [tau * sum(Q[i, c] * K[j, c] for c in range(d)) for j in range(N)]
        z = sum(sp.exp(x) for x in s)
        for c in range(d):
            loss += G[i, c] * sum(sp.exp(s[j]) / z * V[j, c] for j in range(N))
    rng = np.random.default_rng(7)
    vals = {n: rand(rng, N, d) for n in ("Q", "K", "V", "G")}
    U = {n: rand(rng, N, d) for n in ("Q", "K", "V")}
    f = 0
    for n in ("Q", "K", "V"):
        for i in range(N):
            for c in range(d):
                f += U[n][i, c] * sp.diff(loss, sym[n][i, c])
    subs = {sym[n][i, c]: vals[n][i, c] for n in sym for i in range(N) for c in range(d)}
    expect = {n: np.array([[float(sp.diff(f, sym[n][i, c]).evalf(subs=subs, n=30))
                            for c in range(d)] for i in range(N)]) for n in sym}
    ours = orc.attn_bob(vals["Q"], vals["K"], vals["V"], vals["G"], U["Q"], U["K"], U["V"], float(tau))
    for a, n in zip(ours, ("Q", "K", "V", "G")):
        np.testing.assert_allclose(a, expect[n], rtol=1e-11, atol=1e-12)


def test_lemma_e2_closed_form_random():
    """V = dO = UQ = UK = 0, UV = W  =>  ed(dO) = softmax(tau Q K^T) W and the
    other three outputs vanish exactly (evolve.pub review, Strengths: paper
    Lemma E.2)."""
    rng = np.random.default_rng(8)
    N, d, tau = 50, 12, 1.0 / math.sqrt(12)
    Q, K, W = (rand(rng, 2, N, d) for _ in range(3))
    Z = np.zeros_like(Q)
    gQ, gK, gV, gdO = orc.attn_bob(Q, K, Z, Z, Z, Z, W, tau)
    P = scipy.special.softmax(tau * np.einsum("hid,hjd->hij", Q, K), axis=-1)
    np.testing.assert_allclose(gdO, P @ W, rtol=1e-12, atol=1e-13)
    assert not gQ.any() and not gK.any() and not gV.any()


def test_lemma_e2_golden_hand_values():
    with open(os.path.join(GOLDEN, "lemma_e2_hand.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        Q, K, W = (np.array(case[k]) for k in ("Q", "K", "W"))
        Z = np.zeros_like(Q)
        gQ, gK, gV, gdO = orc.attn_bob(Q, K, Z, Z, Z, Z, W, case["tau"])
        np.testing.assert_allclose(gdO, case["expected_gdO"], rtol=0, atol=1e-13)
        assert not gQ.any() and not gK.any() and not gV.any()


# ---------------------------------------------------------------------------
# invariants that hold exactly
# ---------------------------------------------------------------------------

def test_linear_in_upstream_cotangents():
    rng = np.random.default_rng(9)
    N, d, tau = 20, 6, 0.4
    Q, K, V, dO, UQ, UK, UV = inputs(rng, N, d)
    UQ2, UK2, UV2 = (rand(rng, 1, N, d) for _ in range(3))
    a = orc.attn_bob(Q, K, V, dO, UQ, UK, UV, tau)
    b = orc.attn_bob(Q, K, V, dO, UQ2, UK2, UV2, tau)
    c = orc.attn_bob(Q, K, V, dO, 2 * UQ - 3 * UQ2, 2 * UK - 3 * UK2, 2 * UV - 3 * UV2, tau)
    for x, y, z in zip(a, b, c):
        np.testing.assert_allclose(z, 2 * x - 3 * y, rtol=1e-11, atol=1e-12)


def test_uq_uk_zero_gives_zero_gV_and_alpha():
    rng = np.random.default_rng(10)
    N, d, tau = 30, 7, 0.6
    Q, K, V, dO, _, _, UV = inputs(rng, N, d)
    Z = np.zeros_like(Q)
    _, _, gV, _ = orc.attn_bob(Q, K, V, dO, Z, Z, UV, tau)
    alpha, _ = orc.bob_row_scalars(Q, K, V, dO, Z, Z, UV, tau)
    assert not gV.any()
    assert not alpha.any()


def test_key_shift_invariance_column_sums_vanish():
    """g is unchanged by K -> K + 1 c^T and by V -> V + 1 c^T, so the key-side
    BoB outputs sum to zero over keys."""
    rng = np.random.default_rng(11)
    N, d, tau = 33, 9, 0.5
    X = inputs(rng, N, d, H=2)
    _, gK, gV, _ = orc.attn_bob(*X, tau)
    for g in (gK, gV):
        assert np.abs(g.sum(axis=-2)).max() <= 1e-12 * np.abs(g).sum(axis=-2).max()


def test_euler_identities_in_V_and_dO():
    """g is linear in dO and affine-linear in V (dV does not depend on V), so
    <gdO, dO> = f and <gV, V> = <UQ, dQ> + <UK, dK>."""
    rng = np.random.default_rng(12)
    N, d, tau = 27, 8, 0.35
    Q, K, V, dO, UQ, UK, UV = inputs(rng, N, d)
    dQ, dK, dV, _ = orc.attn_bwd(Q, K, V, dO, tau)
    _, _, gV, gdO = orc.attn_bob(Q, K, V, dO, UQ, UK, UV, tau)
    fq, fk, fv = (UQ * dQ).sum(), (UK * dK).sum(), (UV * dV).sum()
    assert abs((gdO * dO).sum() - (fq + fk + fv)) <= 1e-11 * (abs(fq) + abs(fk) + abs(fv))
    assert abs((gV * V).sum() - (fq + fk)) <= 1e-11 * (abs(fq) + abs(fk))


def test_affine_row_scalars_reproduce_row_outputs():
    """The hierarchical affine structure (evolve.pub review, Summary / Key
    claims: paper Prop. 4.1): with alpha, E from ``row_scalars`` the row-side
    outputs follow from alpha-free sums over keys,
        gQ  = tau (dS UK + X K - E (P K) + alpha (Z K)),
        gdO = P UV + (P o B) V - alpha O,
    X = P o (C + B o (dP - D)), Z = P o (2D - dP); and the key-side outputs
    from per-element terms that use alpha and E:
        gK = tau (dS^T UQ + Gs^T Q),  gV = Gdp^T dO,
        Gs = P o (C + B o (dP - D) - E + alpha (2D - dP)),  Gdp = P o (B - alpha).
    """
    rng = np.random.default_rng(13)
    N, d, tau = 40, 8, 0.5
    Q, K, V, dO, UQ, UK, UV = (x[0] for x in inputs(rng, N, d))
    gQ, gK, gV, gdO = orc.bob_rows(Q, K, V, dO, UQ, UK, UV, tau)
    alpha, E = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau)
    S = tau * Q @ K.T
    P = scipy.special.softmax(S, axis=1)
    O = P @ V
    dP = dO @ V.T
    D = (dO * O).sum(1)[:, None]
    B = tau * (UQ @ K.T + Q @ UK.T)
    C = dO @ UV.T
    dS = P * (dP - D)
    X = P * (C + B * (dP - D))
    Z = P * (2 * D - dP)
    a, e = alpha[:, None], E[:, None]
    np.testing.assert_allclose(tau * (dS @ UK + X @ K - e * (P @ K) + a * (Z @ K)), gQ, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(P @ UV + (P * B) @ V - a * O, gdO, rtol=1e-10, atol=1e-12)
    Gs = P * (C + B * (dP - D) - e + a * (2 * D - dP))
    Gdp = P * (B - a)
    np.testing.assert_allclose(tau * (dS.T @ UQ + Gs.T @ Q), gK, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Gdp.T @ dO, gV, rtol=1e-10, atol=1e-12)


def test_row_blocking_matches_single_block(monkeypatch):
    rng = np.random.default_rng(14)
    N, d, tau = 70, 6, 0.5
    X = inputs(rng, N, d, H=2)
    full = orc.attn_bob(*X, tau)
    monkeypatch.setattr(orc, "_BLOCK_ELEMS", 3 * N)      # 3-row blocks, ragged tail
    blocked = orc.attn_bob(*X, tau)
    for a, b in zip(full, blocked):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_sampled_rows_match_full():
    rng = np.random.default_rng(15)
    N, d, tau = 64, 8, 0.5
    X = [x[0] for x in inputs(rng, N, d)]
    gQ, _, _, gdO = orc.attn_bob(*X, tau)
    rows = [0, 5, 63]
    sq, so = orc.bob_sampled_rows(*X, tau, rows)
    np.testing.assert_allclose(sq, gQ[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(so, gdO[rows], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("block_rows,workers", [(None, 1), (5, 3)])
def test_sampled_key_rows_match_full(monkeypatch, block_rows, workers):
    """The key-side sample (every query row swept, sampled key columns kept)
    equals the full sweep's key rows, for whole and for ragged row blocks."""
    rng = np.random.default_rng(16)
    N, d, tau = 64, 8, 0.5
    X = [x[0] for x in inputs(rng, N, d)]
    _, gK, gV, _ = orc.attn_bob(*X, tau)
    _, dK, dV, _ = orc.attn_bwd(*X[:4], tau)
    if block_rows:
        monkeypatch.setattr(orc, "_BLOCK_ELEMS", block_rows * N)
    cols = [0, 1, 31, 62, 63]
    got = orc.bob_sampled_cols(*X, tau, cols, workers=workers)
    for g, ref in zip(got, (dK, dV, gK, gV)):
        np.testing.assert_allclose(g, ref[cols], rtol=1e-12, atol=1e-13)
