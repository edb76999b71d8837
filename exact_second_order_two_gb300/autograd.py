"""Twice-differentiable softmax attention built on the library's three calls.

``attention(q, k, v, causal, scale)`` runs ``fbob_forward``.  Its backward
runs ``fbob_backward``, and the backward of that runs ``fbob_bob``.  So a
second ``torch.autograd.grad`` through a first one taken with
``create_graph=True`` is the exact backward-over-backward of FlashBoB
("FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
Attention", Abstract).  That is the differentiation through the backward pass
that second-order methods, meta-learning and test-time training need, and it
never forms an N x N tensor.

``fbob_bob`` returns the total derivative of <gQ,dQ> + <gK,dK> + <gV,dV>
with respect to Q, K, V and dO, including the paths through O and LSE.
The forward's O and LSE therefore enter the backward node as detached
values, so those paths are not counted a second time.

Every step runs in the CUDA library.  Tensors are [B, H, N, d], contiguous,
bf16 or fp32, on one CUDA device.  There is no CPU path: anything else raises.
"""
from __future__ import annotations

import torch

from . import _binding as _b


def _contig(t: torch.Tensor) -> torch.Tensor:
    return t if t.is_contiguous() else t.contiguous()


class _AttentionBackward(torch.autograd.Function):
    """(q, k, v, dO) -> (dQ, dK, dV); its own backward is fbob_bob."""

    @staticmethod
    def forward(ctx, q, k, v, do, o, lse, causal, scale):
        do = _contig(do)
        dq, dk, dv = _b.backward(q, k, v, o, lse, do, causal, scale)
        ctx.save_for_backward(q, k, v, do, o, lse)
        ctx.causal, ctx.scale = causal, scale
        # a second-order loss that reads only some of dQ, dK, dV leaves the
        # other cotangents None; fbob_bob skips their work
        ctx.set_materialize_grads(False)
        return dq, dk, dv

    @staticmethod
    def backward(ctx, gq, gk, gv):
        q, k, v, do, o, lse = ctx.saved_tensors
        if gq is None and gk is None and gv is None:
            return None, None, None, None, None, None, None, None
        gq, gk, gv = (None if g is None else _contig(g) for g in (gq, gk, gv))
        gradq, gradk, gradv, graddo = _b.bob(q, k, v, o, lse, do, gq, gk, gv,
                                             ctx.causal, ctx.scale)
        return gradq, gradk, gradv, graddo, None, None, None, None


class _Attention(torch.autograd.Function):
    """(q, k, v) -> O = softmax(scale q k^T [+ causal mask]) v."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = _b.forward(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = _AttentionBackward.apply(q, k, v, do, o.detach(), lse.detach(),
                                              ctx.causal, ctx.scale)
        return dq, dk, dv, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: float | None = None) -> torch.Tensor:
    """Softmax attention whose first and second derivatives run in the
    library: O = softmax(scale * q k^T, masked to j <= i when causal) v.

    scale defaults to 1/sqrt(d) and is not differentiated.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise _b.FbobError(1, f"attention: {name} must be a CUDA tensor")
    q, k, v = _contig(q), _contig(k), _contig(v)
    if scale is None:
        scale = 1.0 / float(q.shape[-1]) ** 0.5
    return _Attention.apply(q, k, v, bool(causal), float(scale))
