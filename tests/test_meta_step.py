"""Synthetic second-order workload: one MAML / test-time-training step of an
attention layer (exact_second_order_two_gb300.meta), with the library's
attention against the same step on a dense fp64 CPU attention.

The meta-gradient differentiates through the inner gradient, so the
attention part of it is the backward-over-backward.  The reference writes
softmax attention out densely and lets torch's CPU autograd take its second
derivative.
"""
import numpy as np
import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300.meta import AttentionLayer, layer_forward, maml_step, mse


def dense_attention(q, k, v, causal=True, scale=None):
    """Softmax attention written out, in fp64, with the inputs' rounding."""
    dt = q.dtype
    q, k, v = q.double(), k.double(), v.double()
    if scale is None:
        scale = q.shape[-1] ** -0.5
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        n = q.shape[-2]
        mask = torch.ones(n, n, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, float("-inf"))
    return (torch.softmax(s, dim=-1) @ v).to(dt)


def make_task(B, N, width, seed):
    g = torch.Generator().manual_seed(seed)
    xs, ys, xq, yq = (torch.randn(B, N, width, generator=g) for _ in range(4))
    return (xs, 0.5 * ys), (xq, 0.5 * yq)


def rel(a, b):
    a = a.detach().double().cpu().numpy()
    b = b.detach().double().cpu().numpy()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


LR = 5.0  # large enough that the second-order term is ~10-20% of the meta-gradient


def first_order_meta_grads(layer, support, query, compute):
    """First-order MAML on the dense reference: the inner gradient taken as a
    constant, i.e. without the backward-over-backward term."""
    params = layer.params()
    inner = mse(layer_forward(params, support[0], layer.heads, True, compute, dense_attention),
                support[1])
    g = torch.autograd.grad(inner, params)
    adapted = [w - LR * gi for w, gi in zip(params, g)]
    outer = mse(layer_forward(adapted, query[0], layer.heads, True, compute, dense_attention),
                query[1])
    return torch.autograd.grad(outer, params)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
@pytest.mark.parametrize("compute,tol", [(torch.float32, 1e-3), (torch.bfloat16, 5e-2)],
                         ids=["fp32_cuda_cores", "bf16_tensor_cores"])
def test_maml_step_matches_dense_reference(compute, tol):
    B, N, width, heads = 2, 96, 128, 2
    layer = AttentionLayer.random(width, heads, "cuda", seed=1)
    support, query = make_task(B, N, width, seed=2)
    gpu_task = tuple(tuple(t.cuda() for t in pair) for pair in (support, query))
    loss, grads = maml_step(layer, *gpu_task, inner_lr=LR, compute_dtype=compute)

    ref_layer = AttentionLayer(*(w.detach().double().cpu().requires_grad_(True)
                                 for w in layer.params()), heads=heads)
    cpu_task = tuple(tuple(t.double() for t in pair) for pair in (support, query))
    ref_compute = torch.float64 if compute == torch.float32 else torch.bfloat16
    ref_loss, ref_grads = maml_step(ref_layer, *cpu_task, inner_lr=LR,
                                    compute_dtype=ref_compute, attn=dense_attention)
    assert abs(loss.item() - ref_loss.item()) <= tol * abs(ref_loss.item())
    errs = [rel(g, r) for g, r in zip(grads, ref_grads)]
    assert max(errs) <= tol, errs
    # the comparison can see the second-order term: dropping it (first-order
    # MAML) moves the meta-gradient by more than the tolerance
    fo = first_order_meta_grads(ref_layer, *cpu_task, ref_compute)
    assert max(rel(a, b) for a, b in zip(fo, ref_grads)) > 2 * tol


def test_meta_step_rejects_cpu_attention_inputs():
    layer = AttentionLayer.random(64, 1, "cpu", seed=0)
    support, query = make_task(1, 8, 64, seed=0)
    with pytest.raises(fbob.FbobError):
        maml_step(layer, support, query)
