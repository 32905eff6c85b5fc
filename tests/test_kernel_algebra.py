"""The two-pass schedule the kernels run, restated tile by tile in fp64 NumPy
and checked against the node-by-node reverse-mode oracle (CPU only).

This pins the reformulation the CUDA kernels use (not the oracle): pass 1
accumulates the alpha-free sums U1 = dS UK + X K, U2 = P K, W = dS K and
Y = P UV + (P o B) V over key tiles together with alpha = sum P B and
EX = sum X, and corrects them at the row end,
    gQ = tau (U1 - EX U2 - alpha W),  gdO = Y - alpha O,  E = EX + D alpha;
pass 2 recomputes each tile with the final alpha, E,
    Gs = P (C + (B - alpha) (dP - D) + alpha D - E),  Gdp = P (B - alpha),
    gK = tau (dS^T UQ + Gs^T Q),  gV = Gdp^T dO.
(evolve.pub review, Summary and Key claims: two row scalars alpha, E, two
passes; Strengths: alpha-free accumulators corrected after the reduction.)

The tensor-core pass 1 runs as two sweeps over the same row blocks (TMEM
holds one kernel's accumulators): U1 and Y with alpha and E, writing
gdO = Y - alpha O; then, with EX = E - D alpha read back,
Z = sum_j (EX P + alpha dS) K_j and gQ = tau (U1 - Z).  `two_sweep_pass1`
restates that order; `four_pass_sweeps` restates the four-pass ablation's
three row sweeps the same way.
"""

import numpy as np
import pytest

import oracle.attention as orc


def two_pass(Q, K, V, dO, UQ, UK, UV, tau, L, O, D, br=16, bc=8):
    N, d = Q.shape
    gQ, gdO = np.zeros_like(Q), np.zeros_like(Q)
    alpha, E = np.zeros(N), np.zeros(N)
    for i0 in range(0, N, br):                      # pass 1: row blocks
        r = slice(i0, min(N, i0 + br))
        U1 = np.zeros((r.stop - r.start, d)); U2 = np.zeros_like(U1); W = np.zeros_like(U1); Y = np.zeros_like(U1)
        a = np.zeros(r.stop - r.start); ex = np.zeros_like(a)
        for j0 in range(0, N, bc):                  # loop over key tiles
            c = slice(j0, min(N, j0 + bc))
            P = np.exp(tau * Q[r] @ K[c].T - L[r, None])
            B = tau * (UQ[r] @ K[c].T + Q[r] @ UK[c].T)
            dP = dO[r] @ V[c].T
            C = dO[r] @ UV[c].T
            t = dP - D[r, None]
            dS, X, PB = P * t, P * (C + B * t), P * B
            a += PB.sum(1); ex += X.sum(1)
            U1 += dS @ UK[c] + X @ K[c]; U2 += P @ K[c]; W += dS @ K[c]; Y += P @ UV[c] + PB @ V[c]
        gQ[r] = tau * (U1 - ex[:, None] * U2 - a[:, None] * W)
        gdO[r] = Y - a[:, None] * O[r]
        alpha[r], E[r] = a, ex + D[r] * a
    gK, gV = np.zeros_like(K), np.zeros_like(V)
    for j0 in range(0, N, br):                      # pass 2: key blocks
        c = slice(j0, min(N, j0 + br))
        AK = np.zeros((c.stop - c.start, d)); AV = np.zeros_like(AK)
        for i0 in range(0, N, bc):                  # loop over query tiles
            r = slice(i0, min(N, i0 + bc))
            Pt = np.exp(tau * K[c] @ Q[r].T - L[None, r])
            Bt = tau * (UK[c] @ Q[r].T + K[c] @ UQ[r].T)
            dPt = V[c] @ dO[r].T
            Ct = UV[c] @ dO[r].T
            t = dPt - D[None, r]
            bp = Bt - alpha[None, r]
            dSt = Pt * t
            Gs = Pt * (Ct + bp * t + (alpha * D - E)[None, r])
            Gd = Pt * bp
            AK += dSt @ UQ[r] + Gs @ Q[r]; AV += Gd @ dO[r]
        gK[c], gV[c] = tau * AK, AV
    return gQ, gK, gV, gdO, alpha, E


def two_sweep_pass1(Q, K, V, dO, UQ, UK, UV, tau, L, O, D, br=16, bc=8):
    N, d = Q.shape
    gQ, gdO = np.zeros_like(Q), np.zeros_like(Q)
    ws = np.zeros((N, 2))                           # (alpha, E) per row

    def tiles(r):
        for j0 in range(0, N, bc):
            c = slice(j0, min(N, j0 + bc))
            yield c, np.exp(tau * Q[r] @ K[c].T - L[r, None])

    for i0 in range(0, N, br):                      # sweep 1: U1, Y, alpha, E; gdO = Y - alpha O
        r = slice(i0, min(N, i0 + br))
        n = r.stop - r.start
        U1, Y = np.zeros((n, d)), np.zeros((n, d))
        a, ex = np.zeros(n), np.zeros(n)
        for c, P in tiles(r):
            B = tau * (UQ[r] @ K[c].T + Q[r] @ UK[c].T)
            t = dO[r] @ V[c].T - D[r, None]
            X = P * (dO[r] @ UV[c].T + B * t)
            a += (P * B).sum(1); ex += X.sum(1)
            U1 += (P * t) @ UK[c] + X @ K[c]
            Y += P @ UV[c] + (P * B) @ V[c]
        gQ[r] = U1
        gdO[r] = Y - a[:, None] * O[r]
        ws[r, 0], ws[r, 1] = a, ex + D[r] * a
    for i0 in range(0, N, br):                      # sweep 2: Z, gQ = tau (U1 - Z)
        r = slice(i0, min(N, i0 + br))
        a = ws[r, 0]; ex = ws[r, 1] - D[r] * a
        Z = np.zeros((r.stop - r.start, d))
        for c, P in tiles(r):
            dS = P * (dO[r] @ V[c].T - D[r, None])
            Z += (ex[:, None] * P + a[:, None] * dS) @ K[c]
        gQ[r] = tau * (gQ[r] - Z)
    return gQ, gdO, ws[:, 0], ws[:, 1]


@pytest.mark.parametrize("N,d,sig", [(40, 8, (1,) * 7), (33, 5, (4, 4, 1, 1, 1, 1, 1)), (64, 16, (1, 1, 1, .1, .1, .1, .1))])
def test_two_sweep_pass1_matches_node_by_node_oracle(N, d, sig):
    rng = np.random.default_rng(N * d + 1)
    Q, K, V, dO, UQ, UK, UV = [rng.standard_normal((N, d)) * s for s in sig]
    tau = 1.0 / np.sqrt(d)
    O, L = orc.attn_fwd_head(Q, K, V, tau)
    _, _, _, D = orc.attn_bwd_rows(Q, K, V, dO, tau)
    gQ, gdO, alpha, E = two_sweep_pass1(Q, K, V, dO, UQ, UK, UV, tau, L, O, D)
    ref = orc.bob_rows(Q, K, V, dO, UQ, UK, UV, tau)
    np.testing.assert_allclose(gQ, ref[0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gdO, ref[3], rtol=1e-10, atol=1e-12)
    ra, rE = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau)
    np.testing.assert_allclose(alpha, ra, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(E, rE, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("N,d,sig", [(40, 8, (1,) * 7), (33, 5, (4, 4, 1, 1, 1, 1, 1)), (64, 16, (1, 1, 1, .1, .1, .1, .1))])
def test_two_pass_schedule_matches_node_by_node_oracle(N, d, sig):
    rng = np.random.default_rng(N * d)
    X = [rng.standard_normal((N, d)) * s for s in sig]
    Q, K, V, dO, UQ, UK, UV = X
    tau = 1.0 / np.sqrt(d)
    O, L = orc.attn_fwd_head(Q, K, V, tau)
    _, _, _, D = orc.attn_bwd_rows(Q, K, V, dO, tau)
    got = two_pass(Q, K, V, dO, UQ, UK, UV, tau, L, O, D)
    ref = orc.bob_rows(Q, K, V, dO, UQ, UK, UV, tau)
    for g, r in zip(got[:4], (ref[0], ref[1], ref[2], ref[3])):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)
    alpha, E = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau)
    np.testing.assert_allclose(got[4], alpha, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[5], E, rtol=1e-10, atol=1e-12)


def four_pass_sweeps(Q, K, V, dO, UQ, UK, UV, tau, L, O, D, br=16, bc=8):
    """The four-pass ablation's three row sweeps as the kernels compute them:
    alpha; then E stored as En + 2 alpha D (En = sum_j P Pbar with Pbar =
    tau B (dP - D) + C - alpha dP); then, with En = E - 2 alpha D read back,
    gQ = tau sum_j (dS UK + Sbar K), Sbar = P (Pbar - En), and gdO = Y - alpha O."""
    N, d = Q.shape
    ws = np.zeros((N, 2))
    gQ, gdO = np.zeros_like(Q), np.zeros_like(Q)

    def tiles(r):
        for j0 in range(0, N, bc):
            c = slice(j0, min(N, j0 + bc))
            yield c, np.exp(tau * Q[r] @ K[c].T - L[r, None])

    for i0 in range(0, N, br):                      # sweep 1: alpha
        r = slice(i0, min(N, i0 + br))
        a = np.zeros(r.stop - r.start)
        for c, P in tiles(r):
            a += (P * tau * (UQ[r] @ K[c].T + Q[r] @ UK[c].T)).sum(1)
        ws[r, 0] = a
    for i0 in range(0, N, br):                      # sweep 2: E (natural form, needs alpha)
        r = slice(i0, min(N, i0 + br))
        a = ws[r, 0]
        en = np.zeros(r.stop - r.start)
        for c, P in tiles(r):
            B = tau * (UQ[r] @ K[c].T + Q[r] @ UK[c].T)
            dP = dO[r] @ V[c].T
            en += (P * (B * (dP - D[r, None]) + dO[r] @ UV[c].T - a[:, None] * dP)).sum(1)
        ws[r, 1] = en + 2 * a * D[r]
    for i0 in range(0, N, br):                      # sweep 3: the row outputs, alpha and E known
        r = slice(i0, min(N, i0 + br))
        a = ws[r, 0]
        en = ws[r, 1] - 2 * a * D[r]
        n = r.stop - r.start
        G, Y = np.zeros((n, d)), np.zeros((n, d))
        for c, P in tiles(r):
            B = tau * (UQ[r] @ K[c].T + Q[r] @ UK[c].T)
            dP = dO[r] @ V[c].T
            t = dP - D[r, None]
            Sbar = P * (B * t + dO[r] @ UV[c].T - (a[:, None] * dP + en[:, None]))
            G += (P * t) @ UK[c] + Sbar @ K[c]
            Y += P @ UV[c] + (P * B) @ V[c]
        gQ[r] = tau * G
        gdO[r] = Y - a[:, None] * O[r]
    return gQ, gdO, ws[:, 0], ws[:, 1]


@pytest.mark.parametrize("N,d,sig", [(40, 8, (1,) * 7), (33, 5, (4, 4, 1, 1, 1, 1, 1)), (64, 16, (1, 1, 1, .1, .1, .1, .1))])
def test_four_pass_sweeps_match_node_by_node_oracle(N, d, sig):
    rng = np.random.default_rng(N * d + 3)
    Q, K, V, dO, UQ, UK, UV = [rng.standard_normal((N, d)) * s for s in sig]
    tau = 1.0 / np.sqrt(d)
    O, L = orc.attn_fwd_head(Q, K, V, tau)
    _, _, _, D = orc.attn_bwd_rows(Q, K, V, dO, tau)
    gQ, gdO, alpha, E = four_pass_sweeps(Q, K, V, dO, UQ, UK, UV, tau, L, O, D)
    ref = orc.bob_rows(Q, K, V, dO, UQ, UK, UV, tau)
    # the direct sweep recovers En = E - 2 alpha D by a subtraction that cancels on
    # peaky rows: compare at fp64 rounding of the tensor's scale, not of each element
    np.testing.assert_allclose(gQ, ref[0], rtol=1e-10, atol=1e-10 * np.abs(ref[0]).max())
    np.testing.assert_allclose(gdO, ref[3], rtol=1e-10, atol=1e-10 * np.abs(ref[3]).max())
    ra, rE = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau)
    np.testing.assert_allclose(alpha, ra, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(E, rE, rtol=1e-10, atol=1e-12)   # the workspace form pass 2 reads
