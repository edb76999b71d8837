"""A synthetic second-order workload: one MAML / test-time-training step of a
single attention layer, on random weights.

Test-time training and meta-learning are among the uses of exact
differentiation through the backward pass that FlashBoB names ("FlashBoB:
I/O-Efficient Exact Backward-over-Backward for Softmax Attention",
Abstract).  The layer here is

    y = attention(x Wq, x Wk, x Wv) Wo        (heads split from the width)

The inner step adapts the weights on a support batch:

    W' = W - lr * grad_W L_support(W)         (create_graph=True)

The outer (meta) loss L_query(W') is then differentiated back to W through
that inner gradient.  The attention part of this second derivative is
exactly the library's backward-over-backward: fbob_forward, fbob_backward and
fbob_bob, run through ``attention``.  No N x N tensor is formed at any point.

Only the projections and the losses (plain torch matmuls and reductions)
run outside the library.  They are the workload around the hot path, not part
of it.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from .autograd import attention


@dataclass
class AttentionLayer:
    """Weights of one multi-head attention layer: width = heads * head_dim."""
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    heads: int

    def params(self):
        return [self.wq, self.wk, self.wv, self.wo]

    @staticmethod
    def random(width: int, heads: int, device, dtype=torch.float32, seed: int = 0):
        g = torch.Generator(device="cpu").manual_seed(seed)
        std = width ** -0.5
        ws = [(torch.randn(width, width, generator=g) * std).to(device, dtype)
              for _ in range(4)]
        for w in ws:
            w.requires_grad_(True)
        return AttentionLayer(*ws, heads=heads)


def layer_forward(params, x: torch.Tensor, heads: int, causal: bool = True,
                  compute_dtype=torch.bfloat16, attn=attention) -> torch.Tensor:
    """x: [B, N, width] -> [B, N, width].  Attention runs in `compute_dtype`
    with [B, H, N, d] inputs; the projections run in the weights' dtype."""
    wq, wk, wv, wo = params
    B, N, W = x.shape
    d = W // heads

    def heads_of(t):
        return t.view(B, N, heads, d).transpose(1, 2).contiguous().to(compute_dtype)

    q, k, v = heads_of(x @ wq), heads_of(x @ wk), heads_of(x @ wv)
    o = attn(q, k, v, causal=causal)
    o = o.to(x.dtype).transpose(1, 2).reshape(B, N, W)
    return o @ wo


def mse(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    return ((a - b) ** 2).mean()


def maml_step(layer: AttentionLayer, support, query, inner_lr: float = 0.1,
              causal: bool = True, compute_dtype=torch.bfloat16, attn=attention):
    """One meta-learning step.

    support, query: (x, y) pairs of [B, N, width] tensors.
    Returns (outer_loss, meta_grads): the query loss after one inner SGD step
    on the support loss, and its exact gradient with respect to the
    original weights (second order through the inner gradient).
    """
    params = layer.params()
    xs, ys = support
    xq, yq = query
    inner = mse(layer_forward(params, xs, layer.heads, causal, compute_dtype, attn), ys)
    grads = torch.autograd.grad(inner, params, create_graph=True)
    adapted = [w - inner_lr * g for w, g in zip(params, grads)]
    outer = mse(layer_forward(adapted, xq, layer.heads, causal, compute_dtype, attn), yq)
    meta_grads = torch.autograd.grad(outer, params)
    return outer.detach(), meta_grads
