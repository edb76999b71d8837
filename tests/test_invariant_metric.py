"""The normalised invariant residuals used on GPU outputs separate rounding
noise from real mistakes: exact (oracle) outputs rounded to bf16 score far
below the 0.05 threshold, and outputs with one wrong term score far above."""
import numpy as np
import torch

import oracle
from gpu_helpers import invariant_residuals


def build(n=384, d=32, seed=4, causal=True, wrong=None):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    do, gq, gk, gv = (0.1 * rng.standard_normal((1, 1, n, d)) for _ in range(4))
    scale = 1 / np.sqrt(d)
    dq, dk, dv = oracle.backward_batched(q, k, v, do, causal, scale)
    gradq, gradk, gradv, graddo = oracle.bob_batched(q, k, v, do, gq, gk, gv,
                                                     causal, scale)
    if wrong == "graddo":
        o, _ = oracle.forward_batched(q, k, v, causal, scale)
        graddo = graddo + 0.3 * o          # a mis-weighted r*O term
    if wrong == "gradk":
        gradk = gradk + 0.2 * gk           # a stray term
    t = lambda a: torch.tensor(a).to(torch.bfloat16)  # noqa: E731
    dev = dict(q=t(q), k=t(k), v=t(v), do=t(do), gq=t(gq), gk=t(gk), gv=t(gv))
    return dict(dq=t(dq), dk=t(dk), dv=t(dv), gradq=t(gradq), gradk=t(gradk),
                gradv=t(gradv), graddo=t(graddo), dev=dev)


def test_rounded_exact_outputs_pass():
    res = invariant_residuals(build())
    assert max(res.values()) < 0.01, res


def test_wrong_terms_fail():
    assert invariant_residuals(build(wrong="graddo"))["I1"] > 0.2
    res = invariant_residuals(build(wrong="gradk"))
    assert max(res["I3"], res["I4_gradk"]) > 0.2, res
