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
from gpu_helpers import (FULL_SIZE_SAMPLES, compare_sampled, gpu_pipeline, gpu_sample,
                         invariant_residuals, make, oracle_full, oracle_sample, rel_err,
                         sample_rows, tol_for, to64)

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
        errs = {k: rel_err(to64(gpu[k]), ref[k], floor=zero_floor(ref, k))
                for k in OUTPUTS}
        errs["lse"] = float(np.max(np.abs(to64(gpu["lse"]) - ref["lse"])))
        bad = {k: e for k, e in errs.items() if not e <= (tol if k != "lse" else 1e-2)}
        assert not bad, f"{w.name} path={path}: {bad} (all: {errs})"
        for k in OUTPUTS:
            assert torch.isfinite(gpu[k].float()).all(), k


GROUPS = (("o",), ("dq", "dk", "dv"), ("gradq", "gradk", "gradv", "graddo"))


def zero_floor(ref, key):
    """Denominator floor for an output that is identically zero in exact
    arithmetic (dQ, dK, gradQ, gradK and gradV at N = 1): 10% of the largest
    output of the same call, the scale at which bf16 rounding of the
    cancelled terms is measured.  Every other output is compared against its
    own max|ref| with no floor."""
    group = next(g for g in GROUPS if key in g)
    scale = max(float(np.max(np.abs(ref[k]))) for k in group)
    # fp64 leaves ~1e-17 of the cancelled terms where exact arithmetic gives 0
    if float(np.max(np.abs(ref[key]))) > 1e-9 * scale:
        return None
    return 0.1 * scale


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

def sampled_check(w: Workload, seed=0):
    n_rows, blocks, n_tail = FULL_SIZE_SAMPLES[w.name]
    ins = make(w, seed)
    gpu = gpu_pipeline(ins, w)
    tol = tol_for(w)
    rows = sample_rows(w.N, n_rows, seed + 1)
    checked = set()
    for b, h, c0, nc in blocks:
        x = {k: to64(v[b, h]) for k, v in ins.items()}
        sets = [(rows if (b, h) not in checked else np.array([], dtype=np.int64),
                 np.arange(c0, c0 + nc))]
        if n_tail and (b, h) not in checked:
            sets.append((np.array([], dtype=np.int64), np.arange(w.N - n_tail, w.N)))
        checked.add((b, h))
        for r, c in sets:
            ref = oracle_sample(x, w, r, c)
            got = gpu_sample(gpu, b, h, r, c)
            lse_ref, lse_got = ref.pop("lse", None), got.pop("lse", None)
            bad = compare_sampled(got, ref, tol)
            assert not bad, (w.name, b, h, "cols", int(c[0]) if len(c) else None, bad)
            if lse_ref is not None:
                assert float(np.max(np.abs(lse_got - lse_ref))) <= 1e-2, (w.name, b, h)
    for k in ("gradq", "gradk", "gradv", "graddo"):
        assert torch.isfinite(gpu[k].float()).all(), k
    res = invariant_residuals(gpu)
    assert all(r < 0.05 for r in res.values()), (w.name, res)
    return gpu


@pytest.mark.slow
def test_workload_b2h16_n16384_d128_sampled():
    sampled_check(WORKLOADS["bf16_causal_b2h16_n16384_d128"])


@pytest.mark.slow
def test_workload_peaked_n65536_d128_sampled():
    sampled_check(WORKLOADS["bf16_causal_peaked_h8_n65536_d128"])


@pytest.mark.slow
def test_workload_n262144_d64_sampled():
    sampled_check(WORKLOADS["bf16_causal_h4_n262144_d64"])


@pytest.mark.slow
def test_noncausal_n16384_d128_sampled():
    """Without the mask every tile takes the mask-free path and pass 2
    visits every query tile of every key block (the pass-1 key loop runs to
    N): the long-sequence exact BoB of the paper, not only its causal form."""
    sampled_check(WORKLOADS["bf16_h4_n16384_d128"])


@pytest.mark.slow
@pytest.mark.parametrize("d", [128, 64])
def test_partial_last_head_group(d):
    """The tensor-core kernels visit (batch, head) units in groups of G heads
    (the smallest power of two giving two waves of CTAs per group).  With
    B*H = 3 and 256 row / key blocks per head, G = 2, so the last group holds
    a single head, which takes the partial-group branch of the CTA
    numbering.  Every head is compared with the oracle (sampled rows, the
    last key columns, and an earlier key block of the lone head), and the
    invariants hold on the full outputs."""
    sampled_check(WORKLOADS[f"bf16_causal_b3_n32768_d{d}"], seed=5)


def rows_check(w: Workload, heads, n_rows=12, seed=0):
    """Sampled query rows of a few heads against the oracle, and the exact
    invariants on the full outputs.  Without the mask every key column's
    oracle value needs the row scalars of all N queries (O(N^2 d) per head,
    hours at N=262144), so at these lengths the key-side outputs are held to
    the invariants, which a zeroed or wrong gradK / gradV fails (I2, I3)."""
    ins = make(w, seed)
    gpu = gpu_pipeline(ins, w)
    tol = tol_for(w)
    rows = sample_rows(w.N, n_rows, seed + 1)
    none = np.array([], dtype=np.int64)
    for b, h in heads:
        x = {k: to64(v[b, h]) for k, v in ins.items()}
        ref = oracle_sample(x, w, rows, none)
        got = gpu_sample(gpu, b, h, rows, none)
        lse_ref, lse_got = ref.pop("lse"), got.pop("lse")
        bad = compare_sampled(got, ref, tol)
        assert not bad, (w.name, b, h, bad)
        assert float(np.max(np.abs(lse_got - lse_ref))) <= 1e-2, (w.name, b, h)
    for k in ("gradq", "gradk", "gradv", "graddo"):
        assert torch.isfinite(gpu[k].float()).all(), k
    res = invariant_residuals(gpu)
    assert all(r < 0.05 for r in res.values()), (w.name, res)


@pytest.mark.slow
def test_noncausal_n65536_d128_rows_and_invariants():
    rows_check(WORKLOADS["bf16_h8_n65536_d128"], heads=((0, 0), (0, 5)))


@pytest.mark.slow
def test_noncausal_n262144_d64_rows_and_invariants():
    """The paper's longest length (262K, Abstract) without the mask."""
    rows_check(WORKLOADS["bf16_h4_n262144_d64"], heads=((0, 1), (0, 3)))


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
    # with gV alone, G = 0 and gradV is exactly zero: that output alone is
    # measured against 10% of the call's largest output
    scale = max(float(np.max(np.abs(r))) for r in ref)
    floors = [None if float(np.max(np.abs(r))) > 1e-9 * scale else 0.1 * scale for r in ref]
    tol = tol_for(w)
    errs = [rel_err(to64(g), r, floor=f) for g, r, f in zip(got, ref, floors)]
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
