"""Shared helpers of the GPU parity tests: run the library's fwd -> bwd -> BoB
chain through the C ABI and compare with the fp64 oracle."""

from __future__ import annotations

import numpy as np
import torch

import attn_inputs
import exact_second_order_attn_gb300 as fb
import oracle.attention as orc


def rel_err(gpu, ref):
    """max|gpu - ref| / max|ref| over the whole tensor (0/0 -> max|gpu|)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    num = np.abs(gpu - ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def to_dev(inputs, device="cuda"):
    return {k: v.to(device) for k, v in inputs.items()}


def run_chain(w, inp=None, stream=None, causal=False):
    """Run fwd, bwd and BoB on the GPU; return a dict of CPU float64 arrays."""
    if inp is None:
        inp = attn_inputs.make_inputs(w)
    x = to_dev(inp)
    O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, stream=stream, causal=causal)
    dQ, dK, dV, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau, stream=stream, causal=causal)
    gQ, gK, gV, gdO, ws = fb.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"],
                                      w.tau, stream=stream, causal=causal)
    fb.device_status(stream)
    out = dict(O=O, L=L, dQ=dQ, dK=dK, dV=dV, D=D, gQ=gQ, gK=gK, gV=gV, gdO=gdO,
               alpha=ws[..., 0], E=ws[..., 1])
    return {k: v.double().cpu().numpy() for k, v in out.items()}, inp


def oracle_inputs(inp, heads=None):
    """The same (dtype-rounded) inputs as fp64 numpy arrays, optionally a
    subset of heads as (b, h) pairs."""
    out = {}
    for k, v in inp.items():
        a = v.double().numpy()
        if heads is not None:
            a = np.stack([a[b, h] for b, h in heads])
        out[k] = a
    return out


def oracle_chain(x, tau, causal=False):
    O, L = orc.attn_fwd(x["Q"], x["K"], x["V"], tau, causal=causal)
    dQ, dK, dV, D = orc.attn_bwd(x["Q"], x["K"], x["V"], x["dO"], tau, causal=causal)
    args = [x[k] for k in ("Q", "K", "V", "dO", "UQ", "UK", "UV")]
    gQ, gK, gV, gdO = orc.attn_bob(*args, tau, causal=causal)
    alpha, E = orc.bob_row_scalars(*args, tau, causal=causal)
    return dict(O=O, L=L, dQ=dQ, dK=dK, dV=dV, D=D, gQ=gQ, gK=gK, gV=gV, gdO=gdO, alpha=alpha, E=E)


def select_heads(out, heads):
    return {k: np.stack([v[b, h] for b, h in heads]) for k, v in out.items()}


def cuda_ok():
    return torch.cuda.is_available()
