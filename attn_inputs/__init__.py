"""Seeded synthetic inputs for the attention BoB workloads.

This module only draws random tensors: it holds none of the method's
arithmetic, so both the CUDA path's tests/bench and the CPU oracle can use it.

Recipe (all workloads): one CPU ``torch.Generator`` seeded with ``seed``
draws ``randn`` float32 tensors of shape [B, H, N, d] in the fixed order
Q, K, V, dO, UQ, UK, UV; each is multiplied by its standard deviation and
rounded to the workload's input dtype (bf16: round-to-nearest-even).  The
closed-form case draws Q, K, then W (placed in UV) and sets V, dO, UQ, UK to
zero.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

NAMES = ("Q", "K", "V", "dO", "UQ", "UK", "UV")


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem: shape, dtype, scale and per-tensor std."""
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str                      # "bf16" or "fp32" (inputs); outputs are fp32
    tau: float
    sigma: tuple = (1.0,) * 7       # std of Q, K, V, dO, UQ, UK, UV
    closed_form: bool = False       # V = dO = UQ = UK = 0, UV = W
    seed: int = 0

    @property
    def heads(self) -> int:
        return self.B * self.H

    def with_n(self, N: int) -> "Workload":
        return Workload(self.name.split("@")[0] + f"@N={N}", self.B, self.H, N, self.d,
                        self.dtype, self.tau, self.sigma, self.closed_form, self.seed)


def _long(N):
    return Workload(f"long_context_b1h1_d64@N={N}", 1, 1, N, 64, "bf16", 1.0 / 8.0)


WORKLOADS = {
    # single head, fp32 inputs, full fwd -> bwd -> BoB chain
    "single_head_fp32_b1h1_n256_d64":
        Workload("single_head_fp32_b1h1_n256_d64", 1, 1, 256, 64, "fp32", 1.0 / 8.0),
    # GPT-2-Small-shaped Hessian-estimation step
    "gpt2s_b8h12_n1024_d64":
        Workload("gpt2s_b8h12_n1024_d64", 8, 12, 1024, 64, "bf16", 1.0 / 8.0,
                 (1.0, 1.0, 1.0, 0.1, 0.1, 0.1, 0.1)),
    # long-context sweep, one head
    **{f"long_context_b1h1_d64@N={N}": _long(N) for N in (4096, 16384, 65536, 131072, 262144)},
    # wide heads
    "wide_head_b2h16_n16384_d128":
        Workload("wide_head_b2h16_n16384_d128", 2, 16, 16384, 128, "bf16", 1.0 / math.sqrt(128)),
    # numerics stress: Q, K with std 4 give peaky softmax rows
    "peaky_b4h32_n8192_d128":
        Workload("peaky_b4h32_n8192_d128", 4, 32, 8192, 128, "bf16", 1.0 / math.sqrt(128),
                 (4.0, 4.0, 1.0, 1.0, 1.0, 1.0, 1.0)),
    # profiler case: the wide-head shape with 8 heads (inputs 235 MB > L2)
    "wide_head_b2h4_n16384_d128":
        Workload("wide_head_b2h4_n16384_d128", 2, 4, 16384, 128, "bf16", 1.0 / math.sqrt(128)),
    "long_context_b1h8_n16384_d64":
        Workload("long_context_b1h8_n16384_d64", 1, 8, 16384, 64, "bf16", 1.0 / 8.0),
    # closed-form reduction, fp32
    "closed_form_fp32_b1h1_n32768_d128":
        Workload("closed_form_fp32_b1h1_n32768_d128", 1, 1, 32768, 128, "fp32",
                 1.0 / math.sqrt(128), closed_form=True),
}


def torch_dtype(w: Workload):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[w.dtype]


def make_inputs(w: Workload, pin_memory: bool = False) -> dict:
    """CPU tensors Q, K, V, dO, UQ, UK, UV of shape [B, H, N, d] in the input dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    dt = torch_dtype(w)
    out = {}
    if w.closed_form:
        drawn = {"Q": 1.0, "K": 1.0, "UV": 1.0}
        for name in NAMES:
            if name in drawn:
                t = torch.randn(shape, generator=g, dtype=torch.float32) * drawn[name]
                out[name] = t.to(dt)
            else:
                out[name] = torch.zeros(shape, dtype=dt)
    else:
        for name, s in zip(NAMES, w.sigma):
            t = torch.randn(shape, generator=g, dtype=torch.float32)
            if s != 1.0:
                t.mul_(s)
            out[name] = t.to(dt)
    if pin_memory:
        out = {k: v.pin_memory() for k, v in out.items()}
    return out


def small(B=1, H=1, N=256, d=64, dtype="bf16", tau=None, sigma=(1.0,) * 7, seed=0,
          closed_form=False) -> Workload:
    """An ad-hoc workload for tests (same recipe, any shape)."""
    if tau is None:
        tau = 1.0 / math.sqrt(d)
    return Workload(f"adhoc_b{B}h{H}_n{N}_d{d}_{dtype}", B, H, N, d, dtype, tau,
                    tuple(sigma), closed_form, seed)
