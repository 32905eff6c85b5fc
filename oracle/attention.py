"""Plain fp64 CPU oracle for softmax attention: forward, first backward and
backward-over-backward (BoB).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` use it.  It shares no code with the
CUDA library (no kernels, headers, helpers or constants).

Sources (all four web pages describe one paper, "FlashBoB: I/O-Efficient
Exact Backward-over-Backward for Softmax Attention"):

* abstract (aiqbench.com news item and arxivdaily.com): attention forward and
  first backward in the FlashAttention sense; BoB differentiates through the
  first backward;
* evolve.pub review, "Scope & Claims": BoB is J_g^T applied to upstream
  matrices at (dQ, dK, dV) (paper section 4.1);
* evolve.pub review, FAQ "What is backward-over-backward (BoB)": the
  Jacobian-transpose-vector product of the first-backward map;
* evolve.pub review, FAQ "Is FlashBoB an approximation?": the outputs are
  exact, so the oracle is the plain definition;
* evolve.pub review, Strengths ("Genuinely new algorithmic insight"): the
  paper's Appendix C derives every identity node by node with reverse-mode
  chain rule.  The pages do not print those equations; ``bob_rows`` below is
  that reverse-mode sweep written out for the graph of g, in the order of the
  graph's nodes.

Notation (per head, row-major, rows i = queries, rows j = keys):
    S = tau Q K^T,  P = softmax_row(S),  O = P V,  L_i = logsumexp_j S_ij
    g(Q, K, V, dO) = (dQ, dK, dV) with
        dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),
        dS = P o (dP - D 1^T),  dQ = tau dS K,  dK = tau dS^T Q
    BoB(UQ, UK, UV) = gradient of f = <UQ,dQ> + <UK,dK> + <UV,dV>
        with respect to (Q, K, V, dO)  ->  (gQ, gK, gV, gdO)
        (the pages write these four outputs as ed(Q), ed(K), ed(V), ed(dO)).

Readings where the pages are silent:
* g is a function of (Q, K, V, dO) only; O is not an independent input, so
  D = rowsum(dO o O) is differentiated through O = P V.
* tau multiplies the scores once: S = tau Q K^T.
* L is the natural-log row logsumexp.
* Non-causal attention by default.  The pages never state a mask; with
  ``causal=True`` the plain definition of causal attention is used: query i
  attends to keys j <= i (S_ij = -inf for j > i before the row softmax).
  Every reverse-mode step below multiplies by P, so the masked entries drop
  out of all derivatives without further changes.

Every row of every intermediate (S, P, O, dP, D, dS) depends only on the
query rows of Q and dO of that row, so the graph of g splits exactly into
independent query-row blocks: the query-row outputs (dQ, gQ, gdO, D, L, O)
of a block are complete, and the key-side outputs (dK, dV, gK, gV) are sums
of per-block contributions.  ``_row_blocks`` uses that to bound memory for
long sequences; the arithmetic inside a block is the unblocked definition.

Parity pins (tests/test_oracle_*.py): library softmax/logsumexp, brute force
loops, torch.autograd fp64 first and double backward, a sympy symbolic double
derivative, central finite differences through the adjoint identity, the
closed-form reduction of the evolve.pub review's Strengths item "Theory
honestly scoped" (paper Lemma E.2) and invariants.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "attn_fwd_head",
    "attn_bwd_rows",
    "bob_rows",
    "row_scalars",
    "attn_fwd",
    "attn_bwd",
    "attn_bob",
    "bob_row_scalars",
    "bob_four_pass_rows",
    "attn_bob_four_pass",
    "bob_sampled_rows",
    "bob_sampled_cols",
]

# Largest number of fp64 score elements one row block materialises
# (a block of r rows holds several r x N matrices).
_BLOCK_ELEMS = 1 << 23


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _mask(S: np.ndarray, qidx) -> np.ndarray:
    """Causal mask: S_aj = -inf where key j comes after query qidx[a]
    (qidx None: no mask).  Key 0 is never masked, so every row keeps a
    finite maximum."""
    if qidx is None:
        return S
    keys = np.arange(S.shape[1])
    return np.where(keys[None, :] > np.asarray(qidx)[:, None], -np.inf, S)


def _softmax_rows(S: np.ndarray):
    """Row softmax and natural-log logsumexp with the usual max shift."""
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)
    s = e.sum(axis=1, keepdims=True)
    P = e / s
    L = (m + np.log(s))[:, 0]
    return P, L


# ---------------------------------------------------------------------------
# forward (abstract: FlashAttention-style forward; here materialised)
# ---------------------------------------------------------------------------

def attn_fwd_head(Q, K, V, tau, qidx=None):
    """O = softmax(tau Q K^T) V and L = logsumexp rows, one head, fp64
    (rows of Q are the queries qidx under the causal mask, if given)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    S = _mask(tau * (Q @ K.T), qidx)
    P, L = _softmax_rows(S)
    O = P @ V
    return O, L


# ---------------------------------------------------------------------------
# first backward g (abstract; evolve.pub FAQ "What is backward-over-backward")
# ---------------------------------------------------------------------------

def attn_bwd_rows(Qr, K, V, dOr, tau, qidx=None):
    """First backward restricted to the query rows Qr, dOr of one head
    (query indices qidx under the causal mask, if given).

    Returns (dQ_rows, dK_part, dV_part, D_rows): the row outputs are complete,
    the key-side outputs are this block's contribution to the sums over rows.
    """
    Qr, K, V, dOr = _f64(Qr), _f64(K), _f64(V), _f64(dOr)
    S = _mask(tau * (Qr @ K.T), qidx)
    P, _ = _softmax_rows(S)
    O = P @ V
    dV = P.T @ dOr
    dP = dOr @ V.T
    D = (dOr * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = tau * (dS @ K)
    dK = tau * (dS.T @ Qr)
    return dQ, dK, dV, D


# ---------------------------------------------------------------------------
# backward over backward: reverse mode through the graph of g, node by node
# (evolve.pub review, "Scope & Claims" and Strengths; paper section 4.1 and
# Appendix C)
# ---------------------------------------------------------------------------

def bob_rows(Qr, K, V, dOr, UQr, UK, UV, tau, qidx=None):
    """Reverse-mode sweep of f = <UQ,dQ> + <UK,dK> + <UV,dV> for one query-row
    block of one head (query indices qidx under the causal mask, if given).

    Returns (gQ_rows, gK_part, gV_part, gdO_rows).  Every node of the first
    backward is materialised; adjoints are named ``<node>_bar``.
    """
    Qr, K, V, dOr = _f64(Qr), _f64(K), _f64(V), _f64(dOr)
    UQr, UK, UV = _f64(UQr), _f64(UK), _f64(UV)

    # ---- forward sweep: the nodes of g ---------------------------------
    S = _mask(tau * (Qr @ K.T), qidx)         # S = tau Q K^T (masked)
    P, _ = _softmax_rows(S)                   # P = softmax_row(S)
    O = P @ V                                 # O = P V
    dP = dOr @ V.T                            # dP = dO V^T
    D = (dOr * O).sum(axis=1)                 # D = rowsum(dO o O)
    dS = P * (dP - D[:, None])                # dS = P o (dP - D 1^T)
    # outputs: dQ = tau dS K, dK = tau dS^T Q, dV = P^T dO

    # ---- reverse sweep ---------------------------------------------------
    Q_bar = np.zeros_like(Qr)
    K_bar = np.zeros_like(K)
    V_bar = np.zeros_like(V)
    dO_bar = np.zeros_like(dOr)
    P_bar = np.zeros_like(P)

    # output seeds: dQ_bar = UQ, dK_bar = UK, dV_bar = UV
    # dQ = tau dS K
    dS_bar = tau * (UQr @ K.T)
    K_bar += tau * (dS.T @ UQr)
    # dK = tau dS^T Q
    dS_bar += tau * (Qr @ UK.T)
    Q_bar += tau * (dS @ UK)
    # dV = P^T dO
    P_bar += dOr @ UV.T
    dO_bar += P @ UV
    # dS = P o (dP - D 1^T)
    P_bar += dS_bar * (dP - D[:, None])
    dP_bar = dS_bar * P
    D_bar = -(dS_bar * P).sum(axis=1)
    # D = rowsum(dO o O)
    dO_bar += D_bar[:, None] * O
    O_bar = D_bar[:, None] * dOr
    # dP = dO V^T
    dO_bar += dP_bar @ V
    V_bar += dP_bar.T @ dOr
    # O = P V
    P_bar += O_bar @ V.T
    V_bar += P.T @ O_bar
    # P = softmax_row(S)
    S_bar = P * (P_bar - (P * P_bar).sum(axis=1, keepdims=True))
    # S = tau Q K^T
    Q_bar += tau * (S_bar @ K)
    K_bar += tau * (S_bar.T @ Qr)

    return Q_bar, K_bar, V_bar, dO_bar


def row_scalars(Qr, K, V, dOr, UQr, UK, UV, tau, qidx=None):
    """The two row scalars of the hierarchical affine structure for a row block.

    The pages name them alpha and E (evolve.pub review, Summary and Key claims:
    paper Prop. 4.1) without printing formulas.  Reading used here, with
    B = tau (UQ K^T + Q UK^T) the adjoint reaching dS, C = dO UV^T the adjoint
    reaching P through dV, and dP = dO V^T:

        alpha_i = sum_j P_ij B_ij
        E_i     = sum_j P_ij (C_ij + B_ij dP_ij)

    so that -alpha is the adjoint of D and E - 2 D alpha is the row centre
    rowsum(P o P_bar) of the softmax reverse step in ``bob_rows``.
    """
    Qr, K, V, dOr = _f64(Qr), _f64(K), _f64(V), _f64(dOr)
    UQr, UK, UV = _f64(UQr), _f64(UK), _f64(UV)
    S = _mask(tau * (Qr @ K.T), qidx)
    P, _ = _softmax_rows(S)
    dP = dOr @ V.T
    B = tau * (UQr @ K.T + Qr @ UK.T)
    C = dOr @ UV.T
    alpha = (P * B).sum(axis=1)
    E = (P * (C + B * dP)).sum(axis=1)
    return alpha, E


def bob_four_pass_rows(Qr, K, V, dOr, UQr, UK, UV, tau, qidx=None):
    """BoB of one query-row block computed in the order of the four-pass
    schedule that the affine structure collapses to two (evolve.pub review,
    Strengths: "collapsing a natural four-pass schedule to two").  The pages
    do not spell the four passes out; the reading used here is the order
    plain reverse mode forces when the row scalars are not split off:

      1. alpha_i = sum_j P_ij B_ij (minus the adjoint of D);
      2. En_i = sum_j P_ij Pbar_ij, the centre of the softmax reverse step,
         where Pbar = C + B o (dP - D) - alpha dP needs alpha (the adjoint of
         D reaches P through O = P V);
      3. the row outputs with alpha and En known:
         gQ = tau (dS UK + Sbar K), gdO = P UV + (P o B) V - alpha O,
         Sbar = P o (Pbar - En);
      4. the key-side outputs: gK = tau (dS^T UQ + Sbar^T Q),
         gV = (P o (B - alpha))^T dO.

    B = tau (UQ K^T + Q UK^T) and C = dO UV^T are the adjoints reaching dS
    and (through dV) P, as in ``row_scalars``.  Returns
    (gQ_rows, gK_part, gV_part, gdO_rows, alpha, En).
    """
    Qr, K, V, dOr = _f64(Qr), _f64(K), _f64(V), _f64(dOr)
    UQr, UK, UV = _f64(UQr), _f64(UK), _f64(UV)
    S = _mask(tau * (Qr @ K.T), qidx)
    P, _ = _softmax_rows(S)
    O = P @ V
    dP = dOr @ V.T
    D = (dOr * O).sum(axis=1)
    B = tau * (UQr @ K.T + Qr @ UK.T)
    C = dOr @ UV.T
    # pass 1
    alpha = (P * B).sum(axis=1)
    # pass 2
    P_bar = C + B * (dP - D[:, None]) - alpha[:, None] * dP
    En = (P * P_bar).sum(axis=1)
    # pass 3
    dS = P * (dP - D[:, None])
    S_bar = P * (P_bar - En[:, None])
    gQ = tau * (dS @ UK + S_bar @ K)
    gdO = P @ UV + (P * B) @ V - alpha[:, None] * O
    # pass 4
    gK = tau * (dS.T @ UQr + S_bar.T @ Qr)
    gV = (P * (B - alpha[:, None])).T @ dOr
    return gQ, gK, gV, gdO, alpha, En


# ---------------------------------------------------------------------------
# batched drivers over [..., N, d] arrays
# ---------------------------------------------------------------------------

def _row_blocks(N: int):
    r = max(1, min(N, _BLOCK_ELEMS // max(N, 1)))
    for s in range(0, N, r):
        yield slice(s, min(N, s + r))


def _heads(x):
    x = _f64(x)
    lead = x.shape[:-2]
    return x.reshape((-1,) + x.shape[-2:]), lead


def _qidx(rows, causal):
    return np.arange(rows.start, rows.stop) if causal else None


def attn_fwd(Q, K, V, tau, causal=False):
    """O [..., N, d], L [..., N] for every head of [..., N, d] inputs."""
    Qh, lead = _heads(Q)
    Kh, _ = _heads(K)
    Vh, _ = _heads(V)
    O = np.empty(Qh.shape[:-1] + (Vh.shape[-1],))
    L = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for rows in _row_blocks(Qh.shape[1]):
            O[h, rows], L[h, rows] = attn_fwd_head(Qh[h, rows], Kh[h], Vh[h], tau, _qidx(rows, causal))
    return O.reshape(lead + O.shape[1:]), L.reshape(lead + L.shape[1:])


def attn_bwd(Q, K, V, dO, tau, causal=False):
    """(dQ, dK, dV, D) for every head of [..., N, d] inputs."""
    Qh, lead = _heads(Q)
    Kh, _ = _heads(K)
    Vh, _ = _heads(V)
    dOh, _ = _heads(dO)
    dQ = np.empty_like(Qh)
    dK = np.zeros_like(Kh)
    dV = np.zeros_like(Vh)
    D = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for rows in _row_blocks(Qh.shape[1]):
            q, k, v, dd = attn_bwd_rows(Qh[h, rows], Kh[h], Vh[h], dOh[h, rows], tau, _qidx(rows, causal))
            dQ[h, rows] = q
            dK[h] += k
            dV[h] += v
            D[h, rows] = dd
    shp = lambda a: a.reshape(lead + a.shape[1:])
    return shp(dQ), shp(dK), shp(dV), shp(D)


def attn_bob(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """(gQ, gK, gV, gdO) for every head of [..., N, d] inputs."""
    Qh, lead = _heads(Q)
    Kh, _ = _heads(K)
    Vh, _ = _heads(V)
    dOh, _ = _heads(dO)
    UQh, _ = _heads(UQ)
    UKh, _ = _heads(UK)
    UVh, _ = _heads(UV)
    gQ = np.empty_like(Qh)
    gK = np.zeros_like(Kh)
    gV = np.zeros_like(Vh)
    gdO = np.empty_like(dOh)
    for h in range(Qh.shape[0]):
        for rows in _row_blocks(Qh.shape[1]):
            q, k, v, o = bob_rows(Qh[h, rows], Kh[h], Vh[h], dOh[h, rows],
                                  UQh[h, rows], UKh[h], UVh[h], tau, _qidx(rows, causal))
            gQ[h, rows] = q
            gK[h] += k
            gV[h] += v
            gdO[h, rows] = o
    shp = lambda a: a.reshape(lead + a.shape[1:])
    return shp(gQ), shp(gK), shp(gV), shp(gdO)


def bob_row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """(alpha, E) [..., N] for every head (see ``row_scalars``)."""
    Qh, lead = _heads(Q)
    Kh, _ = _heads(K)
    Vh, _ = _heads(V)
    dOh, _ = _heads(dO)
    UQh, _ = _heads(UQ)
    UKh, _ = _heads(UK)
    UVh, _ = _heads(UV)
    alpha = np.empty(Qh.shape[:-1])
    E = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for rows in _row_blocks(Qh.shape[1]):
            alpha[h, rows], E[h, rows] = row_scalars(
                Qh[h, rows], Kh[h], Vh[h], dOh[h, rows], UQh[h, rows], UKh[h], UVh[h], tau, _qidx(rows, causal))
    return alpha.reshape(lead + alpha.shape[1:]), E.reshape(lead + E.shape[1:])


def attn_bob_four_pass(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """(gQ, gK, gV, gdO, alpha, En) for every head, in the four-pass order
    (see ``bob_four_pass_rows``)."""
    Qh, lead = _heads(Q)
    Kh, _ = _heads(K)
    Vh, _ = _heads(V)
    dOh, _ = _heads(dO)
    UQh, _ = _heads(UQ)
    UKh, _ = _heads(UK)
    UVh, _ = _heads(UV)
    gQ = np.empty_like(Qh)
    gK = np.zeros_like(Kh)
    gV = np.zeros_like(Vh)
    gdO = np.empty_like(dOh)
    alpha = np.empty(Qh.shape[:-1])
    En = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for rows in _row_blocks(Qh.shape[1]):
            q, k, v, o, a, e = bob_four_pass_rows(Qh[h, rows], Kh[h], Vh[h], dOh[h, rows],
                                                  UQh[h, rows], UKh[h], UVh[h], tau, _qidx(rows, causal))
            gQ[h, rows] = q
            gK[h] += k
            gV[h] += v
            gdO[h, rows] = o
            alpha[h, rows] = a
            En[h, rows] = e
    shp = lambda a: a.reshape(lead + a.shape[1:])
    return shp(gQ), shp(gK), shp(gV), shp(gdO), shp(alpha), shp(En)


def bob_sampled_rows(Q, K, V, dO, UQ, UK, UV, tau, rows, causal=False):
    """Query-row outputs (gQ, gdO) of one head restricted to the given rows.

    The row-side outputs of a row are complete from that row alone (see the
    module docstring), so long sequences can be checked on a sample of rows.
    """
    rows = np.asarray(rows)
    gQ, _, _, gdO = bob_rows(_f64(Q)[rows], K, V, _f64(dO)[rows], _f64(UQ)[rows], UK, UV, tau,
                             rows if causal else None)
    return gQ, gdO


def _bob_cols_block(Q, K, V, dO, UQ, UK, UV, tau, cols, rows, causal):
    """One query-row block's contribution to the key-side outputs at the key
    rows ``cols`` (see ``bob_sampled_cols``)."""
    qidx = _qidx(rows, causal)
    Qr, dOr, UQr = Q[rows], dO[rows], UQ[rows]
    # forward sweep over every key: the row reductions need whole rows
    S = _mask(tau * (Qr @ K.T), qidx)
    P, _ = _softmax_rows(S)
    O = P @ V
    dP = dOr @ V.T
    D = (dOr * O).sum(axis=1)
    # reverse sweep of bob_rows up to its two row reductions
    dS_bar = tau * (UQr @ K.T + Qr @ UK.T)         # from the dQ and dK seeds
    D_bar = -(dS_bar * P).sum(axis=1)
    O_bar = D_bar[:, None] * dOr
    # P_bar = dO UV^T + dS_bar o (dP - D) + O_bar V^T, with O_bar V^T = D_bar dP
    P_bar = dOr @ UV.T + dS_bar * (dP - D[:, None]) + D_bar[:, None] * dP
    centre = (P * P_bar).sum(axis=1)
    # the rest of the sweep acts entry by entry: keep only the sampled keys
    Pj, dPj, dS_barj, P_barj = P[:, cols], dP[:, cols], dS_bar[:, cols], P_bar[:, cols]
    dSj = Pj * (dPj - D[:, None])
    S_barj = Pj * (P_barj - centre[:, None])
    dP_barj = dS_barj * Pj
    dK = tau * (dSj.T @ Qr)
    dV = Pj.T @ dOr
    gK = tau * (dSj.T @ UQr) + tau * (S_barj.T @ Qr)
    gV = dP_barj.T @ dOr + Pj.T @ O_bar
    return dK, dV, gK, gV


def bob_sampled_cols(Q, K, V, dO, UQ, UK, UV, tau, cols, causal=False, workers=1):
    """Key-side outputs (dK, dV, gK, gV) of one head restricted to the key rows
    ``cols``.

    A key row's outputs are sums over all query rows, and each query row's
    term needs three reductions over all of that row's keys: the softmax
    normaliser, D, and in the reverse sweep of ``bob_rows`` the adjoint of D
    (minus alpha) and the centre rowsum(P o P_bar) of the softmax reverse step.
    So every query-row block is swept over all keys up to those reductions; the
    remaining steps act on single entries and are taken on the sampled key
    columns only before the contraction over the block's query rows.
    ``workers`` > 1 runs the independent row blocks on that many threads; the
    partial sums are added in block order either way.
    """
    cols = np.asarray(cols)
    args = tuple(_f64(a) for a in (Q, K, V, dO, UQ, UK, UV))
    blocks = list(_row_blocks(args[0].shape[0]))
    run = lambda rows: _bob_cols_block(*args, tau, cols, rows, causal)
    if workers > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(workers) as ex:
            parts = list(ex.map(run, blocks))
    else:
        parts = [run(rows) for rows in blocks]
    out = [np.zeros((len(cols), a.shape[1])) for a in (args[1], args[2], args[1], args[2])]
    for part in parts:
        for o, p in zip(out, part):
            o += p
    return tuple(out)
