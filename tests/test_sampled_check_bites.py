"""The sampled comparison used at the full sizes catches wrong outputs.

At N >= 16384 the GPU outputs are compared with the fp64 oracle on sampled
query rows and key columns only, each set against its own max|ref|.  Here the
same comparison runs on the host: the oracle's own outputs (rounded to bf16,
as the GPU returns them) pass it, and a zeroed dK, dV, gradK or gradV, or a
gradQ off by 5%, each fail it, even with cotangents scaled so small that
every output is far below the 1e-2 absolute floor an earlier version of the
check divided by.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (BF16_TOL, FULL_SIZE_SAMPLES, compare_sampled, oracle_sample,
                         rel_err, sample_rows)
from exact_second_order_two_gb300.synthetic import WORKLOADS, Workload

W = Workload("bites", 1, 1, 640, 32, "bf16", True, 1.0, 1.0, 1e-3)


def bf16(a):
    return torch.tensor(a).to(torch.bfloat16).double().numpy()


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(7)
    names = ("q", "k", "v", "do", "gq", "gk", "gv")
    x = {n: bf16(rng.standard_normal((W.N, W.d)) * (1.0 if n in "qkv" else W.cot_std))
         for n in names}
    rows = sample_rows(W.N, 12, 3)
    cols = np.arange(0, 64)
    ref = oracle_sample(x, W, rows, cols)
    ref.pop("lse")
    # what a correct kernel returns: the exact outputs at bf16 precision
    full = dict(zip(("gradq", "gradk", "gradv", "graddo"),
                    oracle.bob(*(x[n] for n in names), W.causal, W.scale)))
    full["o"], _ = oracle.forward(x["q"], x["k"], x["v"], W.causal, W.scale)
    full["dq"], full["dk"], full["dv"] = oracle.backward(x["q"], x["k"], x["v"], x["do"],
                                                         W.causal, W.scale)
    got = {}
    for k in ("gradq", "graddo", "o", "dq"):
        got[k] = bf16(full[k][rows])
    for k in ("gradk", "gradv", "dk", "dv"):
        got[k] = bf16(full[k][cols])
    return got, ref


def test_outputs_are_tiny(case):
    _, ref = case
    # every BoB output is below the old absolute floor
    for k in ("gradq", "gradk", "gradv", "graddo"):
        assert np.max(np.abs(ref[k])) < 1e-2, k


def test_correct_outputs_pass(case):
    got, ref = case
    assert compare_sampled(got, ref, BF16_TOL) == {}


@pytest.mark.parametrize("name", ["gradk", "gradv", "dk", "dv"])
def test_zeroed_key_side_output_fails(case, name):
    got, ref = case
    bad = dict(got, **{name: np.zeros_like(got[name])})
    assert name in compare_sampled(bad, ref, BF16_TOL)


def test_five_percent_off_gradq_fails(case):
    got, ref = case
    bad = dict(got, gradq=got["gradq"] * 1.05)
    assert "gradq" in compare_sampled(bad, ref, BF16_TOL)


def test_identically_zero_reference_needs_a_floor():
    with pytest.raises(ValueError):
        rel_err(np.zeros(3), np.zeros(3))
    assert rel_err(np.full(3, 1e-4), np.zeros(3), floor=1e-2) == pytest.approx(1e-2)


def test_full_size_samples_use_key_blocks_with_real_gradient():
    """Every full-size workload compares at least one key block that is not
    at the end of the sequence: one seen by at least a thousand queries."""
    for name, (n_rows, blocks, _) in FULL_SIZE_SAMPLES.items():
        w = WORKLOADS[name]
        assert n_rows >= 12
        for b, h, c0, nc in blocks:
            assert 0 <= b < w.B and 0 <= h < w.H
            assert 0 <= c0 and c0 + nc <= w.N
            seen_by = w.N - (c0 + nc - 1) if w.causal else w.N
            assert seen_by >= 1000, (name, c0)
