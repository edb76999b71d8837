"""Autograd integration: torch.autograd through fbob_forward -> fbob_backward
-> fbob_bob, against the fp64 oracle.

A first torch.autograd.grad with create_graph=True gives (dQ, dK, dV).  A
second grad of L = <gQ,dQ> + <gK,dK> + <gV,dV> with respect to (Q, K, V, dO)
is BoB.  Both must match the oracle on the same dtype-rounded inputs.
"""
import numpy as np
import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300.synthetic import Workload

import oracle
from gpu_helpers import BF16_TOL, FP32_TOL, make, rel_err, to64

gpu = [pytest.mark.gpu,
       pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

CASES = [
    # name,              B, H,   N,   d, dtype, causal
    ("bf16_causal_ragged", 1, 2, 200, 128, "bf16", True),
    ("bf16_full_d64",      2, 1, 130,  64, "bf16", False),
    ("fp32_causal",        1, 1,  96,  64, "fp32", True),
]


def test_attention_rejects_cpu_tensors():
    x = torch.zeros(1, 1, 4, 64)
    with pytest.raises(fbob.FbobError):
        fbob.attention(x, x, x)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_double_backward_matches_oracle(case):
    name, B, H, N, d, dtype, causal = case
    w = Workload(name, B, H, N, d, dtype, causal, 1.0, 1.0, 0.3)
    ins = make(w, seed=3)
    dev = {k: v.cuda() for k, v in ins.items()}
    q, k, v = (dev[n].clone().requires_grad_() for n in ("q", "k", "v"))
    do = dev["do"].clone().requires_grad_()
    o = fbob.attention(q, k, v, causal=causal)
    dq, dk, dv = torch.autograd.grad(o, (q, k, v), do, create_graph=True)
    L = sum((g.float() * x.float()).sum() for g, x in
            ((dev["gq"], dq), (dev["gk"], dk), (dev["gv"], dv)))
    gradq, gradk, gradv, graddo = torch.autograd.grad(L, (q, k, v, do))
    torch.cuda.synchronize()

    x = {n: to64(t) for n, t in ins.items()}
    ref_o, _ = oracle.forward_batched(x["q"], x["k"], x["v"], causal, w.scale)
    ref_b = oracle.backward_batched(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
    ref_bob = oracle.bob_batched(x["q"], x["k"], x["v"], x["do"], x["gq"], x["gk"],
                                 x["gv"], causal, w.scale)
    tol = FP32_TOL if dtype == "fp32" else BF16_TOL
    got = {"o": o, "dq": dq, "dk": dk, "dv": dv, "gradq": gradq, "gradk": gradk,
           "gradv": gradv, "graddo": graddo}
    ref = {"o": ref_o, "dq": ref_b[0], "dk": ref_b[1], "dv": ref_b[2],
           "gradq": ref_bob[0], "gradk": ref_bob[1], "gradv": ref_bob[2],
           "graddo": ref_bob[3]}
    errs = {n: rel_err(to64(got[n]), ref[n]) for n in got}
    assert all(e <= tol for e in errs.values()), errs


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_unused_cotangents_are_zero():
    """Only dK feeds the second-order loss: autograd hands fbob_bob zero gQ
    and gV, and the result equals BoB with those cotangents zeroed."""
    w = Workload("bf16_gk_only", 1, 2, 160, 64, "bf16", True, 1.0, 1.0, 0.3)
    ins = make(w, seed=5)
    dev = {k: v.cuda() for k, v in ins.items()}
    q, k, v = (dev[n].clone().requires_grad_() for n in ("q", "k", "v"))
    do = dev["do"].clone().requires_grad_()
    o = fbob.attention(q, k, v, causal=True)
    _, dk, _ = torch.autograd.grad(o, (q, k, v), do, create_graph=True)
    L = (dev["gk"].float() * dk.float()).sum()
    grads = torch.autograd.grad(L, (q, k, v, do))
    x = {n: to64(t) for n, t in ins.items()}
    z = np.zeros_like(x["gq"])
    ref = oracle.bob_batched(x["q"], x["k"], x["v"], x["do"], z, x["gk"], z, True, w.scale)
    errs = [rel_err(to64(g), r) for g, r in zip(grads, ref)]
    assert max(errs) <= BF16_TOL, errs
