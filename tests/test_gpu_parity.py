"""GPU parity: the library's fwd -> bwd -> BoB chain (through the C ABI)
against the fp64 oracle on the same seeded inputs, element by element.

Tolerances (per output tensor, max|gpu - ref| / max|ref|):
* bf16 inputs: 1e-2 (fp32 accumulation; the tensor-core path rounds the
  on-chip P-type operands to bf16, which bounds the error near 2^-8
  relative per product before averaging);
* fp32 inputs: 2e-5 for the full chain (fp32 FMA everywhere), and 1e-5 on
  the closed-form reduction (evolve.pub review, Strengths: paper Lemma E.2).
"""

import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
import oracle.attention as orc
from exact_second_order_attn_gb300.build import build
from gpu_helpers import oracle_chain, oracle_inputs, rel_err, run_chain, select_heads, to_dev

pytestmark = pytest.mark.gpu

BF16_TOL = 1e-2
FP32_TOL = 2e-5
CLOSED_FORM_TOL = 1e-5
KEYS = ("O", "L", "dQ", "dK", "dV", "D", "gQ", "gK", "gV", "gdO", "alpha", "E")
# Peaked softmax rows (Q, K with std 4) are where bf16 operand roundings meet
# cancellations (dP - D and Y - alpha O on a row's dominant key); those seeds
# are held to 0.7 of the bf16 bar so that the margin is visible.
PEAKY_MARGIN_TOL = 0.7 * BF16_TOL
# Identity residuals at any size: <gdO, dO> - f and <gV, V> - (<UQ,dQ> + <UK,dK>)
# are random-sign sums of per-element errors, and so are the reference sums,
# so their ratio is of the order of the per-element relative error: bf16
# operand rounding (unit roundoff 2^-9) on the tensor-core path.  They are held
# to the bf16 parity bar.
IDENTITY_TOL = BF16_TOL


def log_errors(case, errs):
    """Append measured errors to $FBOB_PARITY_LOG (one JSON line per case)."""
    path = os.environ.get("FBOB_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **{k: float(v) for k, v in errs.items()}}) + "\n")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    fb.load()
    torch.cuda.init()


def compare_all(gpu, ref, tol, keys=KEYS, case=None):
    errs = {k: rel_err(gpu[k], ref[k]) for k in keys}
    log_errors(case or os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], errs)
    bad = {k: e for k, e in errs.items() if not (e <= tol)}
    assert not bad, f"over tolerance {tol}: {bad} (all: {errs})"
    return errs


def test_single_head_fp32_full_chain():
    w = attn_inputs.WORKLOADS["single_head_fp32_b1h1_n256_d64"]
    gpu, inp = run_chain(w)
    compare_all(gpu, oracle_chain(oracle_inputs(inp), w.tau), FP32_TOL)


@pytest.mark.parametrize("B,H,N,d,sigma", [
    (1, 1, 128, 64, (1,) * 7),
    (2, 3, 384, 64, (1,) * 7),
    (1, 2, 256, 128, (1,) * 7),
    (1, 1, 640, 128, (1,) * 7),
    (1, 2, 512, 128, (4, 4, 1, 1, 1, 1, 1)),
    (2, 1, 256, 64, (1, 1, 1, .1, .1, .1, .1)),
])
def test_bf16_small_shapes(B, H, N, d, sigma):
    w = attn_inputs.small(B, H, N, d, "bf16", sigma=sigma, seed=N + d)
    gpu, inp = run_chain(w)
    compare_all(gpu, oracle_chain(oracle_inputs(inp), w.tau), BF16_TOL)


@pytest.mark.parametrize("N,d", [(200, 64), (37, 128), (1, 64), (33, 64)])
def test_fp32_ragged_and_degenerate(N, d):
    w = attn_inputs.small(1, 2, N, d, "fp32", seed=N)
    gpu, inp = run_chain(w)
    ref = oracle_chain(oracle_inputs(inp), w.tau)
    if N == 1:
        # one key: the softmax is constant, dS = 0 and gQ = gK = 0 exactly
        for k in ("gQ", "gK", "dQ", "dK"):
            assert np.abs(gpu[k]).max() <= 1e-6 * max(1.0, np.abs(ref["gdO"]).max())
        keys = ("O", "L", "dV", "D", "gV", "gdO", "alpha", "E")
    else:
        keys = KEYS
    compare_all(gpu, ref, FP32_TOL, keys)


def test_gpt2s_hessian_step_shape():
    w = attn_inputs.WORKLOADS["gpt2s_b8h12_n1024_d64"]
    gpu, inp = run_chain(w)
    compare_all(gpu, oracle_chain(oracle_inputs(inp), w.tau), BF16_TOL)


@pytest.mark.parametrize("N", [4096, 16384])
def test_long_context_full(N):
    w = attn_inputs.WORKLOADS[f"long_context_b1h1_d64@N={N}"]
    gpu, inp = run_chain(w)
    compare_all(gpu, oracle_chain(oracle_inputs(inp), w.tau), BF16_TOL)


def sampled_row_checks(w, gpu, inp, rows, head=(0, 0)):
    """Row-side outputs on sampled rows against the oracle (the row outputs of
    a query row need only that row), plus exact-math properties of the key
    side that hold at any size."""
    b, h = head
    x = {k: v[b, h].double().numpy() for k, v in inp.items()}
    g = {k: v[b, h] for k, v in gpu.items()}
    rows = np.asarray(rows)
    O, L = orc.attn_fwd_head(x["Q"][rows], x["K"], x["V"], w.tau)
    dQ, _, _, D = orc.attn_bwd_rows(x["Q"][rows], x["K"], x["V"], x["dO"][rows], w.tau)
    args = [x[k] for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV")]
    gQ, gdO = orc.bob_sampled_rows(*args, w.tau, rows)
    alpha, E = orc.row_scalars(x["Q"][rows], x["K"], x["V"], x["dO"][rows], x["UQ"][rows], x["UK"], x["UV"], w.tau)
    ref = dict(O=O, L=L, dQ=dQ, D=D, gQ=gQ, gdO=gdO, alpha=alpha, E=E)
    errs = {k: rel_err(g[k][rows], v) for k, v in ref.items()}
    assert all(e <= BF16_TOL for e in errs.values()), errs
    # key-shift invariance: gK, gV and dK sum to zero over keys
    for k in ("gK", "gV", "dK"):
        colsum = np.abs(g[k].sum(axis=0)).max()
        scale = np.abs(g[k]).sum(axis=0).max()
        assert colsum <= 1e-3 * scale, (k, colsum, scale)
    # dV sums to the column sums of dO over keys
    np.testing.assert_allclose(g["dV"].sum(axis=0), x["dO"].sum(axis=0), rtol=1e-3,
                               atol=1e-3 * np.abs(x["dO"]).sum(axis=0).max())
    # Euler identities: <gdO, dO> = f, <gV, V> = <UQ, dQ> + <UK, dK>
    fq = (x["UQ"] * g["dQ"]).sum()
    fk = (x["UK"] * g["dK"]).sum()
    fv = (x["UV"] * g["dV"]).sum()
    mag = abs(fq) + abs(fk) + abs(fv)
    r1 = abs((g["gdO"] * x["dO"]).sum() - (fq + fk + fv)) / mag
    r2 = abs((g["gV"] * x["V"]).sum() - (fq + fk)) / (abs(fq) + abs(fk))
    log_errors(os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0] + ":identities",
               {**errs, "euler_gdO": r1, "euler_gV": r2})
    assert r1 <= IDENTITY_TOL and r2 <= IDENTITY_TOL, (r1, r2)
    return errs


@pytest.mark.parametrize("N", [65536, 131072, 262144])
def test_long_context_sampled_rows(N):
    w = attn_inputs.WORKLOADS[f"long_context_b1h1_d64@N={N}"]
    gpu, inp = run_chain(w)
    rows = [0, 1, 127, 128, N // 2 + 3, N - 129, N - 1]
    sampled_row_checks(w, gpu, inp, rows)


def test_long_context_sampled_key_rows():
    """Key-side outputs (dK, dV, gK, gV) at N = 65536 element by element on
    sampled key rows: tile edges, the middle and the last rows.  A key row's
    outputs sum over every query row, so the oracle sweeps all query rows up
    to their row reductions and keeps only the sampled keys after that."""
    N = 65536
    w = attn_inputs.WORKLOADS[f"long_context_b1h1_d64@N={N}"]
    gpu, inp = run_chain(w)
    x = {k: v[0, 0].double().numpy() for k, v in inp.items()}
    cols = [0, 1, 127, 128, N // 2 + 3, N - 129, N - 1]
    args = [x[k] for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV")]
    ref = orc.bob_sampled_cols(*args, w.tau, cols, workers=os.cpu_count() or 1)
    errs = {k: rel_err(gpu[k][0, 0][cols], r) for k, r in zip(("dK", "dV", "gK", "gV"), ref)}
    log_errors("long_context_sampled_key_rows", errs)
    assert all(e <= BF16_TOL for e in errs.values()), errs


@pytest.mark.parametrize("name,heads,seed", [
    ("wide_head_b2h16_n16384_d128", [(0, 0), (1, 15)], 0),
    ("peaky_b4h32_n8192_d128", [(0, 0), (3, 31)], 0),
    ("peaky_b4h32_n8192_d128", [(1, 7), (2, 20)], 1),
    ("peaky_b4h32_n8192_d128", [(0, 31), (3, 0)], 2),
])
def test_d128_workloads_sampled_heads(name, heads, seed):
    w = dataclasses.replace(attn_inputs.WORKLOADS[name], seed=seed)
    gpu, inp = run_chain(w)
    ref = oracle_chain(oracle_inputs(inp, heads), w.tau)
    tol = PEAKY_MARGIN_TOL if name.startswith("peaky") else BF16_TOL
    compare_all(select_heads(gpu, heads), ref, tol, case=f"{name}:seed{seed}")
    # every head: finite, and the exact key-side properties
    for k, v in gpu.items():
        assert np.isfinite(v).all(), k
    sampled_row_checks(w, gpu, inp, [0, w.N // 2, w.N - 1], head=(w.B - 1, w.H // 2))


def test_closed_form_fp32():
    """V = dO = UQ = UK = 0, UV = W: gdO = softmax(tau Q K^T) W, the other
    three outputs vanish (evolve.pub review, Strengths: paper Lemma E.2)."""
    w = attn_inputs.WORKLOADS["closed_form_fp32_b1h1_n32768_d128"]
    gpu, inp = run_chain(w)
    x = oracle_inputs(inp)
    expect, _ = orc.attn_fwd(x["Q"], x["K"], x["UV"], w.tau)
    err = rel_err(gpu["gdO"], expect)
    log_errors("closed_form_fp32", {"gdO": err})
    assert err <= CLOSED_FORM_TOL
    for k in ("gQ", "gK", "gV"):
        assert not np.any(gpu[k]), k
    rows = [0, 4097, w.N - 1]
    args = [x[k][0, 0] for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV")]
    _, gdo_rows = orc.bob_sampled_rows(*args, w.tau, rows)
    assert rel_err(gpu["gdO"][0, 0][rows], gdo_rows) <= CLOSED_FORM_TOL


def test_empty_problems_launch_nothing():
    """B*H*N == 0 is a valid problem: every call returns OK and the library's
    per-launch records show that nothing was launched."""
    torch.cuda.synchronize()
    fb.fbob_profile_report()              # drop earlier records
    was = fb.fbob_profile_enable(True)
    try:
        for shape in ((0, 2, 128, 64), (1, 1, 0, 64), (2, 0, 256, 128)):
            for dt in (torch.bfloat16, torch.float32):
                Q = torch.zeros(shape, dtype=dt, device="cuda")
                O, L = fb.attn_fwd(Q, Q, Q, 0.125)
                dQ, dK, dV, D = fb.attn_bwd(Q, Q, Q, O, Q, L, 0.125)
                fb.attn_bob(Q, Q, Q, O, Q, L, D, Q, Q, Q, 0.125)
                assert O.numel() == 0 and L.numel() == 0 and dQ.numel() == 0
        fb.device_status()
        report = fb.fbob_profile_report()
    finally:
        fb.fbob_profile_enable(was)
    assert report == {}, report


def test_no_nxn_allocation_and_static_memory():
    """The library allocates nothing: peak memory over a BoB call is the
    caller's tensors only, at a size where one N x N fp32 matrix is 16 GiB."""
    w = attn_inputs.WORKLOADS["long_context_b1h1_d64@N=65536"]
    x = to_dev(attn_inputs.make_inputs(w))
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau)
    dQ, dK, dV, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau)
    outs = [torch.empty_like(O) for _ in range(4)]
    ws = torch.empty(w.B, w.H, w.N, 2, device="cuda")
    args = (x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau, *outs, ws)
    fb.attn_bob(*args)  # warm (module load)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    fb.attn_bob(*args)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() == base
    assert free0 - free1 < (1 << 20)
    assert ws.numel() * 4 == fb.bob_workspace_bytes(x["Q"]) == 8 * w.N


def test_non_default_stream_and_repeatability():
    w = attn_inputs.small(2, 2, 256, 64, "bf16", seed=3)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, inp = run_chain(w, stream=s)
    b, _ = run_chain(w, inp)
    for k in KEYS:
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 3, 320, 64, False), (2, 3, 200, 128, True), (8, 12, 1024, 64, False)])
def test_head_groups_match_per_batch_calls(B, H, N, d, causal):
    """Every head's first backward and BoB depend on that head alone, so one
    call over B x H heads (which the library may run as two head groups on two
    streams when a launch's last wave would be mostly empty) must equal, bit
    for bit, one call per batch entry (a different grouping, or none)."""
    w = attn_inputs.small(B, H, N, d, "bf16", seed=31)
    x = {k: v.cuda() for k, v in attn_inputs.make_inputs(w).items()}
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, causal=causal)
    _, _, _, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, causal=causal)
    names = ("Q", "K", "V", "O", "dO", "L", "D", "UQ", "UK", "UV")
    full = dict(x, O=O, L=L, D=D)
    whole = fb.attn_bob(*(full[k] for k in names), w.tau, causal=causal)
    whole_bwd = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, causal=causal)
    for b in range(B):
        one = fb.attn_bob(*(full[k][b:b + 1].contiguous() for k in names), w.tau, causal=causal)
        for i, name in enumerate(("gQ", "gK", "gV", "gdO", "ws")):
            assert torch.equal(whole[i][b:b + 1], one[i]), (name, b)
        sl = {k: full[k][b:b + 1].contiguous() for k in ("Q", "K", "V", "O", "dO", "L")}
        one_bwd = fb.attn_bwd(sl["Q"], sl["K"], sl["V"], sl["O"], sl["dO"], sl["L"], w.tau, causal=causal)
        for i, name in enumerate(("dQ", "dK", "dV", "D")):
            assert torch.equal(whole_bwd[i][b:b + 1], one_bwd[i]), (name, b)
    fb.device_status()


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 3, 320, 64, False), (2, 3, 200, 128, True)])
def test_bob_replays_in_a_cuda_graph(B, H, N, d, causal):
    """fbob_attn_bob and fbob_attn_bob_noalloc captured in a CUDA graph (after a
    first eager call in the context, as the header asks) replay to the eager
    results bit for bit - including the two-stream head groups these shapes
    take, whose fork and join must be capture-legal."""
    w = attn_inputs.small(B, H, N, d, "bf16", seed=43)
    x = {k: v.cuda() for k, v in attn_inputs.make_inputs(w).items()}
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, causal=causal)
    _, _, _, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, causal=causal)
    args = (x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau)
    outs = [torch.empty_like(O) for _ in range(4)] + [torch.empty(B, H, N, 2, device="cuda")]
    nouts = [torch.empty_like(O) for _ in range(4)]
    fb.fbob_attn_bob(*args, *outs, causal=causal)
    fb.fbob_attn_bob_noalloc(*args, *nouts, causal=causal)
    torch.cuda.synchronize()
    ref, nref = [t.clone() for t in outs], [t.clone() for t in nouts]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fb.fbob_attn_bob(*args, *outs, causal=causal)
        fb.fbob_attn_bob_noalloc(*args, *nouts, causal=causal)
    for t in outs + nouts:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    fb.device_status()
    for a, b in zip(outs + nouts, ref + nref):
        assert torch.equal(a, b)


def test_wide_head_causal_sampled_heads():
    """The causal bench configuration (B=2, H=16, N=16384, d=128, causal) at
    full size, every output against the causal oracle on two sampled heads."""
    w = attn_inputs.WORKLOADS["wide_head_b2h16_n16384_d128"]
    heads = [(0, 3), (1, 12)]
    gpu, inp = run_chain(w, causal=True)
    ref = oracle_chain(oracle_inputs(inp, heads), w.tau, causal=True)
    compare_all(select_heads(gpu, heads), ref, BF16_TOL, case="wide_head_b2h16_n16384_d128:causal")
