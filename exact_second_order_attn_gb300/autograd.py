"""PyTorch autograd integration: attention that can be differentiated twice.

``attention(Q, K, V, tau)`` returns O = softmax(tau Q K^T) V.  Its backward
runs the library's first backward (dQ, dK, dV), and that backward is itself
differentiable: its vector-Jacobian product - the backward-over-backward -
runs ``fbob_attn_bob``.  So ``torch.autograd.grad(..., create_graph=True)``
followed by a second ``grad`` gives Hessian-vector products of any loss built
on this attention, the use the FlashBoB pages lead with (evolve.pub review,
Summary and Key claims: Hessian-vector products through attention for
second-order optimisers such as Sophia-H).

Exactly as in the kernels' C ABI:
* Q, K, V are bf16 (tensor-core kernels) or fp32 (FFMA kernels), any N;
  O, dQ, dK, dV and the second-order outputs are fp32;
* the incoming gradient of O and the cotangents of dQ, dK, dV are rounded to
  the input dtype before they reach the kernels (the kernels read them at the
  input precision);
* gradients returned for Q, K, V are cast back to the input dtype.

BoB is J_g^T U for g(Q, K, V, dO) = (dQ, dK, dV), with O and L recomputed
from (Q, K, V) inside g: the saved O and L therefore enter the backward node
detached, and no gradient flows into them.  Third derivatives are not
provided.

Every computation runs in the library; this module only moves tensors
between autograd and the binding.
"""

from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import _lib


def _as(t: torch.Tensor | None, like: torch.Tensor) -> torch.Tensor:
    if t is None:
        return torch.zeros_like(like)
    return t.to(like.dtype).contiguous()


class _AttnBwd(torch.autograd.Function):
    """(Q, K, V, dO) -> (dQ, dK, dV); its own backward is BoB."""

    @staticmethod
    def forward(ctx, Q, K, V, dO, O, L, tau, causal):
        dQ, dK, dV, D = _lib.fbob_attn_bwd(Q, K, V, O, dO, L, tau, causal=causal)
        ctx.save_for_backward(Q, K, V, dO, O, L, D)
        ctx.tau, ctx.causal = tau, causal
        return dQ, dK, dV

    @staticmethod
    @once_differentiable
    def backward(ctx, UQ, UK, UV):
        Q, K, V, dO, O, L, D = ctx.saved_tensors
        gQ, gK, gV, gdO, _ = _lib.fbob_attn_bob(Q, K, V, O, dO, L, D, _as(UQ, Q), _as(UK, Q), _as(UV, Q), ctx.tau,
                                                causal=ctx.causal)
        return gQ.to(Q.dtype), gK.to(K.dtype), gV.to(V.dtype), gdO.to(dO.dtype), None, None, None, None


class _Attn(torch.autograd.Function):
    """(Q, K, V) -> O; its backward is the differentiable _AttnBwd."""

    @staticmethod
    def forward(ctx, Q, K, V, tau, causal):
        O, L = _lib.fbob_attn_fwd(Q, K, V, tau, causal=causal)
        ctx.save_for_backward(Q, K, V, O, L)
        ctx.tau, ctx.causal = tau, causal
        return O

    @staticmethod
    def backward(ctx, gO):
        Q, K, V, O, L = ctx.saved_tensors
        dO = _as(gO, Q)
        dQ, dK, dV = _AttnBwd.apply(Q, K, V, dO, O.detach(), L.detach(), ctx.tau, ctx.causal)
        return dQ.to(Q.dtype), dK.to(K.dtype), dV.to(V.dtype), None, None


def attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, tau: float, causal: bool = False) -> torch.Tensor:
    """O = softmax(tau Q K^T) V for [B, H, N, d] tensors, twice differentiable
    (``causal``: query i attends to keys j <= i)."""
    if not (Q.is_contiguous() and K.is_contiguous() and V.is_contiguous()):
        raise ValueError("Q, K, V must be contiguous")
    return _Attn.apply(Q, K, V, float(tau), bool(causal))


def hvp(loss_fn, params, vectors):
    """Hessian-vector product of ``loss_fn(*params)`` (a scalar) in the
    direction ``vectors``, by double backward: returns H v per parameter."""
    params = [p if p.requires_grad else p.detach().requires_grad_(True) for p in params]
    loss = loss_fn(*params)
    grads = torch.autograd.grad(loss, params, create_graph=True)
    dot = sum((g.float() * v.float()).sum() for g, v in zip(grads, vectors))
    return torch.autograd.grad(dot, params)
