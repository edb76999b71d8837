"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs.

Small and ragged shapes are checked element by element on every output; the
five reference workloads are checked in full where the oracle finishes in
seconds, and on sampled rows / tail columns plus exact invariants at the
full sizes the benchmark runs.  Tolerance: max|err| / max|ref| <= 2e-2 for
bf16 inputs and <= 1e-4 for fp32 inputs.
"""
import numpy as np
import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300.synthetic import WORKLOADS, Workload

import oracle
from gpu_helpers import (gpu_pipeline, invariant_residuals, make, oracle_full,
                         rel_err, sample_rows, tol_for, to64)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

OUTPUTS = ("o", "dq", "dk", "dv", "gradq", "gradk", "gradv", "graddo")


def check_full(w: Workload, seed=0, paths=(None,)):
    ins = make(w, seed)
    ref = oracle_full(ins, w)
    for path in paths:
        old = fbob.force_path(-1 if path is None else path)
        try:
            gpu = gpu_pipeline(ins, w)
        finally:
            fbob.force_path(old)
        tol = tol_for(w)
        errs = {k: rel_err(to64(gpu[k]), ref[k], floor=group_floor(ref, k))
                for k in OUTPUTS}
        errs["lse"] = float(np.max(np.abs(to64(gpu["lse"]) - ref["lse"])))
        bad = {k: e for k, e in errs.items() if not e <= (tol if k != "lse" else 1e-2)}
        assert not bad, f"{w.name} path={path}: {bad} (all: {errs})"
        for k in OUTPUTS:
            assert torch.isfinite(gpu[k].float()).all(), k


GROUPS = (("o",), ("dq", "dk", "dv"), ("gradq", "gradk", "gradv", "graddo"))


def group_floor(ref, key):
    """Denominator floor for outputs that vanish in exact arithmetic (e.g.
    gradQ and gradK at N = 1): 10% of the largest output of the same call,
    the scale at which bf16 rounding of the cancelled terms is measured."""
    group = next(g for g in GROUPS if key in g)
    return 0.1 * max(float(np.max(np.abs(ref[k]))) for k in group)


SMALL = [
    # name,            B, H,   N,   d, dtype, causal
    ("fp32_tiny",      1, 1,   1,  64, "fp32", True),
    ("fp32_ragged",    2, 1,  37,  40, "fp32", True),
    ("fp32_noncausal", 1, 2, 129, 128, "fp32", False),
    ("bf16_one",       1, 1,   1,  64, "bf16", True),
    ("bf16_d64",       1, 2, 300,  64, "bf16", True),
    ("bf16_d64_nc",    2, 1, 200,  64, "bf16", False),
    ("bf16_d128",      2, 1, 257, 128, "bf16", True),
    ("bf16_d128_nc",   1, 1, 129, 128, "bf16", False),
    ("bf16_d40",       1, 2,  77,  40, "bf16", True),
    ("bf16_d128_long", 1, 1, 1000, 128, "bf16", True),
    # several key blocks and query tiles without the mask, a ragged last
    # 128-key forward tile (1000 = 7*128 + 104) and two (batch, head) units
    ("bf16_d128_nc_long", 1, 2, 1000, 128, "bf16", False),
    ("bf16_d64_nc_long",  2, 1, 1000, 64, "bf16", False),
    ("bf16_d64_long",     1, 1, 1000, 64, "bf16", True),
]


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_small_shapes_match_oracle(spec):
    name, B, H, N, d, dt, causal = spec
    w = Workload(name, B, H, N, d, dt, causal, 1.0, 1.0, 0.5 if dt == "bf16" else 1.0)
    check_full(w, seed=N)


def test_nondefault_scale():
    w = Workload("scale", 1, 2, 190, 64, "bf16", True, 1.0, 1.0, 0.3)
    ins = make(w, 3)
    scale = 0.37
    x = {k: to64(v) for k, v in ins.items()}
    ref = oracle.bob_batched(x["q"], x["k"], x["v"], x["do"], x["gq"], x["gk"],
                             x["gv"], True, scale)
    d = {k: v.cuda() for k, v in ins.items()}
    o, lse = fbob.forward(d["q"], d["k"], d["v"], True, scale)
    got = fbob.bob(d["q"], d["k"], d["v"], o, lse, d["do"], d["gq"], d["gk"], d["gv"],
                   True, scale)
    for g, r in zip(got, ref):
        assert rel_err(to64(g), r) <= 2e-2


def test_workload_fp32_n256_full():
    check_full(WORKLOADS["fp32_n256_d64"])


def test_workload_bf16_n4096_full():
    check_full(WORKLOADS["bf16_causal_h8_n4096_d64"])


def test_both_kernel_families_agree_with_oracle():
    w = Workload("paths", 1, 2, 333, 128, "bf16", True, 1.0, 1.0, 0.3)
    check_full(w, seed=5, paths=(fbob.PATH_SIMT, None))


def test_invariants_small():
    w = Workload("inv", 2, 2, 512, 64, "bf16", True, 1.0, 1.0, 0.1)
    gpu = gpu_pipeline(make(w, 9), w)
    for k, r in invariant_residuals(gpu).items():
        assert r < 0.05, (k, r)


# ---------------------------------------------------- full-size workloads ---

def sampled_check(w: Workload, n_rows=24, n_tail=128, heads=((0, 0),), seed=0):
    ins = make(w, seed)
    gpu = gpu_pipeline(ins, w)
    tol = tol_for(w)
    rows = sample_rows(w.N, n_rows, seed + 1)
    cols = np.arange(w.N - n_tail, w.N)
    for b, h in heads:
        x = {k: to64(v[b, h]) for k, v in ins.items()}
        args = (x["q"], x["k"], x["v"], x["do"], x["gq"], x["gk"], x["gv"],
                w.causal, w.scale)
        gq_r, gdo_r = oracle.bob_rows(*args, rows)
        gk_c, gv_c = oracle.bob_cols(*args, cols)
        # the forward and first backward that produced BoB's inputs, sampled
        # the same way
        fb = (x["q"], x["k"], x["v"])
        o_r, lse_r = oracle.forward_rows(*fb, w.causal, w.scale, rows)
        dq_r = oracle.backward_rows(*fb, x["do"], w.causal, w.scale, rows)
        dk_c, dv_c = oracle.backward_cols(*fb, x["do"], w.causal, w.scale, cols)
        got = {"gradq": to64(gpu["gradq"][b, h])[rows],
               "graddo": to64(gpu["graddo"][b, h])[rows],
               "gradk": to64(gpu["gradk"][b, h])[cols],
               "gradv": to64(gpu["gradv"][b, h])[cols],
               "o": to64(gpu["o"][b, h])[rows],
               "dq": to64(gpu["dq"][b, h])[rows],
               "dk": to64(gpu["dk"][b, h])[cols],
               "dv": to64(gpu["dv"][b, h])[cols]}
        ref = {"gradq": gq_r, "graddo": gdo_r, "gradk": gk_c, "gradv": gv_c,
               "o": o_r, "dq": dq_r, "dk": dk_c, "dv": dv_c}
        errs = {k: rel_err(got[k], ref[k]) for k in got}
        assert all(e <= tol for e in errs.values()), (w.name, b, h, errs)
        lse_err = float(np.max(np.abs(to64(gpu["lse"][b, h])[rows] - lse_r)))
        assert lse_err <= 1e-2, (w.name, b, h, lse_err)
    for k in ("gradq", "gradk", "gradv", "graddo"):
        assert torch.isfinite(gpu[k].float()).all(), k
    res = invariant_residuals(gpu)
    assert all(r < 0.05 for r in res.values()), (w.name, res)
    return gpu


@pytest.mark.slow
def test_workload_b2h16_n16384_d128_sampled():
    w = WORKLOADS["bf16_causal_b2h16_n16384_d128"]
    sampled_check(w, heads=((0, 0), (1, 15)))


@pytest.mark.slow
def test_workload_peaked_n65536_d128_sampled():
    w = WORKLOADS["bf16_causal_peaked_h8_n65536_d128"]
    sampled_check(w, heads=((0, 3),), n_tail=64)


@pytest.mark.slow
def test_workload_n262144_d64_sampled():
    w = WORKLOADS["bf16_causal_h4_n262144_d64"]
    sampled_check(w, n_rows=12, n_tail=32, heads=((0, 1),))


# ------------------------------------------------- optional cotangents ---

SUBSETS = [("gq",), ("gk",), ("gv",), ("gq", "gk"), ("gq", "gv"), ("gk", "gv")]


@pytest.mark.parametrize("present", SUBSETS, ids=["+".join(p) for p in SUBSETS])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "bf16"), (40, "fp32")],
                         ids=["d64_tc", "d128_tc", "d40_simt"])
def test_absent_cotangents_are_zero(present, d, dtype):
    """gq / gk / gv passed as None (NULL in the C ABI): the result equals BoB
    with those cotangents zero, on both kernel families."""
    w = Workload("opt", 1, 2, 193, d, dtype, True, 1.0, 1.0, 0.3)
    ins = make(w, 11)
    x = {k: to64(v) for k, v in ins.items()}
    zero = np.zeros_like(x["gq"])
    cot = {n: (x[n] if n in present else zero) for n in ("gq", "gk", "gv")}
    ref = oracle.bob_batched(x["q"], x["k"], x["v"], x["do"], cot["gq"], cot["gk"], cot["gv"],
                             True, w.scale)
    dev = {k: v.cuda() for k, v in ins.items()}
    o, lse = fbob.forward(dev["q"], dev["k"], dev["v"], True, w.scale)
    got = fbob.bob(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                   *(dev[n] if n in present else None for n in ("gq", "gk", "gv")),
                   True, w.scale)
    floor = 0.1 * max(float(np.max(np.abs(r))) for r in ref)
    tol = tol_for(w)
    errs = [rel_err(to64(g), r, floor=floor) for g, r in zip(got, ref)]
    assert max(errs) <= tol, (present, errs)


def test_all_cotangents_absent_gives_zeros():
    w = Workload("none", 1, 1, 70, 64, "bf16", True, 1.0, 1.0, 0.3)
    dev = {k: v.cuda() for k, v in make(w, 2).items()}
    o, lse = fbob.forward(dev["q"], dev["k"], dev["v"], True, w.scale)
    outs = tuple(torch.full_like(dev["q"], float("nan")) for _ in range(4))
    got = fbob.bob(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], None, None, None, True,
                   w.scale, out=outs)
    for g in got:
        assert torch.count_nonzero(g).item() == 0
