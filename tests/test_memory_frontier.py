"""Memory frontier: exact BoB through dense PyTorch double-backward needs
memory quadratic in N (it materialises P and the other N x N intermediates).
FlashBoB's never forms an N x N tensor ("FlashBoB: I/O-Efficient Exact
Backward-over-Backward for Softmax Attention", Abstract), so its memory is
linear in N.

On CPU: the library's workspace is linear in N.  On the GPU (slow): the
dense baseline's peak memory is measured at small N and fitted; the fit
predicts where it runs out of memory on this device (it is never driven
there); fbob_bob runs at N = 262,144 and at N = 1,048,576 with peak memory
linear in N.
"""
import ctypes
import math

import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300 import _binding as B


def test_workspace_is_linear_in_n():
    for op in (fbob.OP_BACKWARD, fbob.OP_BOB):
        sizes = []
        for n in (65536, 131072, 262144):
            s = B.make_shape(1, 4, n, 64, torch.bfloat16, True, 0.125)
            sizes.append(B.lib().fbob_workspace_size(op, ctypes.byref(s)))
        assert abs(sizes[1] / sizes[0] - 2) < 1e-3 and abs(sizes[2] / sizes[1] - 2) < 1e-3
    # the N = 262,144, H = 4, d = 64 BoB workspace: about 0.3 GB, nowhere
    # near the 4 * 262144^2 * 4 bytes = 1.1 TB of one fp32 N x N tensor per head
    assert sizes[2] < 0.35e9


def dense_bob(q, k, v, do, gq, gk, gv, causal=True):
    """Exact BoB by torch double-backward of softmax attention written out
    densely (fp32, N x N scores)."""
    scale = q.shape[-1] ** -0.5
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        n = q.shape[-2]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool, device=q.device).triu(1),
                          float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    dq, dk, dv = torch.autograd.grad(o, (q, k, v), do, create_graph=True)
    L = (gq * dq).sum() + (gk * dk).sum() + (gv * dv).sum()
    return torch.autograd.grad(L, (q, k, v, do))


def peak_bytes(fn):
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    fn()
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base


def inputs(n, d, dtype, grad=False):
    g = torch.Generator(device="cpu").manual_seed(n)
    t = [(torch.randn(1, 1, n, d, generator=g) * (1.0 if i < 3 else 0.1)).to("cuda", dtype)
         for i in range(7)]
    if grad:
        for x in t[:4]:
            x.requires_grad_(True)
    return t


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_dense_baseline_is_quadratic_and_fbob_is_linear(capsys):
    d = 128
    dense = {}
    for n in (1024, 2048, 4096):
        t = inputs(n, d, torch.float32, grad=True)
        dense[n] = peak_bytes(lambda: dense_bob(*t))
        del t
    # quadratic growth: doubling N multiplies the dense peak by ~4
    assert dense[4096] / dense[2048] > 3.5
    per_n2 = dense[4096] / 4096 ** 2           # bytes per score element per head
    total = torch.cuda.get_device_properties(0).total_memory
    n_oom_head = int(math.sqrt(total / per_n2))         # one (batch, head)
    n_oom_bench = int(math.sqrt(total / (32 * per_n2)))  # B*H = 32

    fb = {}
    for n in (65536, 262144, 1048576):
        q, k, v, do, gq, gk, gv = inputs(n, d if n < 1048576 else 64, torch.bfloat16)
        o, lse = fbob.forward(q, k, v, True)
        fb[n] = peak_bytes(lambda: fbob.bob(q, k, v, o, lse, do, gq, gk, gv, True))
        assert torch.isfinite(fbob.bob(q, k, v, o, lse, do, gq, gk, gv, True)[0].float()).all()
        del q, k, v, do, gq, gk, gv, o, lse
    # linear growth: 4x N costs ~4x memory at the same d, far from 16x
    assert fb[262144] / fb[65536] < 4.5
    with capsys.disabled():
        print(f"\n[frontier] dense fp32 BoB peak: {dense} bytes; {per_n2:.1f} B per N^2 per head; "
              f"predicted OOM on {total / 2**30:.0f} GiB: N ~ {n_oom_head} for one head, "
              f"N ~ {n_oom_bench} at B*H = 32")
        print(f"[frontier] fbob_bob peak (B=H=1; d=128, d=64 at 1M): {fb} bytes")
