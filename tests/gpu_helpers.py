"""Helpers for the GPU tests: run the CUDA path through the C ABI, run the
oracle on the same (dtype-rounded) inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300.synthetic import Workload, make_inputs

import oracle

BF16_TOL = 2e-2   # max|err| / max|ref| for bf16 inputs
FP32_TOL = 1e-4   # max|err| / max|ref| for fp32 inputs


def tol_for(w: Workload) -> float:
    return FP32_TOL if w.dtype == "fp32" else BF16_TOL


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, ref, floor: float | None = None) -> float:
    """max|got - ref| / max|ref| over the compared elements.

    There is no absolute floor by default: the error of every compared set is
    measured against that set's own largest reference value, so an output
    that is small everywhere (late key columns under a causal mask, say) is
    held to the same relative tolerance as a large one, and a zero or a
    perturbed output fails.  ``floor`` is only for sets that are exactly zero
    in exact arithmetic (gradQ and gradK at N = 1, causal row 0), where only
    rounding noise of cancelled terms is left; the caller then passes the
    scale that noise is measured against."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = float(np.max(np.abs(ref))) if ref.size else 0.0
    if floor is not None:
        denom = max(denom, floor)
    if denom == 0.0:
        raise ValueError("reference is identically zero: pass the floor its "
                         "rounding noise is measured against")
    return float(np.max(np.abs(got - ref)) / denom)


def compare_sampled(got: dict, ref: dict, tol: float) -> dict:
    """Relative errors of sampled output sets (each set against its own
    max|ref|); returns {name: error} for the sets above ``tol``."""
    errs = {name: rel_err(got[name], ref[name]) for name in ref}
    return {name: e for name, e in errs.items() if not e <= tol}


def gpu_pipeline(ins: dict, w: Workload, device="cuda"):
    """forward -> backward -> BoB on the GPU, all through the C ABI."""
    d = {k: v.to(device) for k, v in ins.items()}
    o, lse = fbob.forward(d["q"], d["k"], d["v"], w.causal, w.scale)
    dq, dk, dv = fbob.backward(d["q"], d["k"], d["v"], o, lse, d["do"],
                               w.causal, w.scale)
    grads = fbob.bob(d["q"], d["k"], d["v"], o, lse, d["do"], d["gq"], d["gk"],
                     d["gv"], w.causal, w.scale)
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, gradq=grads[0],
                gradk=grads[1], gradv=grads[2], graddo=grads[3], dev=d)


def oracle_full(ins: dict, w: Workload):
    """Full fp64 oracle on the dtype-rounded inputs, per (b, h)."""
    x = {k: to64(v) for k, v in ins.items()}
    o, lse = oracle.forward_batched(x["q"], x["k"], x["v"], w.causal, w.scale)
    dq, dk, dv = oracle.backward_batched(x["q"], x["k"], x["v"], x["do"],
                                         w.causal, w.scale)
    gq, gk, gv, gdo = oracle.bob_batched(x["q"], x["k"], x["v"], x["do"], x["gq"],
                                         x["gk"], x["gv"], w.causal, w.scale)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, gradq=gq, gradk=gk, gradv=gv,
                graddo=gdo)


def invariant_residuals(gpu: dict):
    """Normalised residuals of the exact BoB invariants on GPU outputs.

    Each identity <a,b> = c is reported as |<a,b> - c| / sqrt(sum (a*b)^2 +
    ...): the size a rounding error of relative size eps produces is ~eps,
    while a wrong term produces ~1.
      I1  <graddO, dO> = L
      I2  <gradV, V>  = <gQ,dQ> + <gK,dK>
      I3  <gradQ, Q> - <gradK, K> = <gK,dK> - <gQ,dQ>
      I4  sum_j gradK_j = 0 and sum_j gradV_j = 0 per (b, h)
    with L = <gQ,dQ> + <gK,dK> + <gV,dV> from the GPU's first backward.
    """
    f = lambda t: t.double()  # noqa: E731
    dv_ = gpu["dev"]

    def ip(a, b):
        prod = f(a) * f(b)
        return prod.sum().item(), torch.sqrt((prod * prod).sum()).item()

    gq_dq, s1 = ip(dv_["gq"], gpu["dq"])
    gk_dk, s2 = ip(dv_["gk"], gpu["dk"])
    gv_dv, s3 = ip(dv_["gv"], gpu["dv"])
    L = gq_dq + gk_dk + gv_dv
    a1, t1 = ip(gpu["graddo"], dv_["do"])
    a2, t2 = ip(gpu["gradv"], dv_["v"])
    a3q, t3q = ip(gpu["gradq"], dv_["q"])
    a3k, t3k = ip(gpu["gradk"], dv_["k"])
    res = {
        "I1": abs(a1 - L) / (t1 + s1 + s2 + s3),
        "I2": abs(a2 - (gq_dq + gk_dk)) / (t2 + s1 + s2),
        "I3": abs((a3q - a3k) - (gk_dk - gq_dq)) / (t3q + t3k + s1 + s2),
    }
    for name in ("gradk", "gradv"):
        g = f(gpu[name])
        col_sum = g.sum(dim=2)                              # [B, H, d]
        col_scale = torch.sqrt((g * g).sum(dim=2))
        res["I4_" + name] = (col_sum.abs() / col_scale.clamp_min(1e-30)).max().item()
    return res


# Full-size samples.  Row-local outputs (O, LSE, dQ, gradQ, graddO) are
# compared on random query rows plus rows 0, N/2 and N - 1.  Key-side outputs
# (dK, dV, gradK, gradV) are compared on a block of key columns chosen to
# carry real gradient and to run pass 2's long query loops (key block 0 is
# seen by every query; a mid block by half of them), plus the last columns
# (the shortest loops) as a set of their own.  Each set is measured against
# its own max|ref|: there is no absolute floor.  The oracle's cost for a key
# block is that of every query row that sees it, so the blocks at N >= 65536
# sit where a few thousand queries see them.
#   workload: (rows sampled, [(b, h, first key column, key columns)], tail)
FULL_SIZE_SAMPLES = {
    "bf16_causal_b2h16_n16384_d128": (24, [(0, 0, 0, 128), (1, 15, 8256, 64)], 64),
    "bf16_causal_peaked_h8_n65536_d128": (16, [(0, 3, 65536 - 4096, 128)], 64),
    "bf16_causal_h4_n262144_d64": (12, [(0, 1, 262144 - 1152, 64)], 32),
    # no mask: every query sees every key, so one block (across the key
    # block boundary at 8192) costs a full head
    "bf16_h4_n16384_d128": (16, [(0, 2, 8192 - 32, 64)], 0),
    # B*H = 3 at N = 32768: heads taken in groups of two, the last group
    # holding one head; every head is sampled
    "bf16_causal_b3_n32768_d128": (12, [(b, 0, 32768 - 1088, 64) for b in range(3)], 32),
    "bf16_causal_b3_n32768_d64": (12, [(b, 0, 32768 - 1088, 64) for b in range(3)], 32),
}


def oracle_sample(x, w: Workload, rows, cols):
    """fp64 oracle values of every output at query rows ``rows`` and key
    columns ``cols`` of one (batch, head) slice ``x``."""
    args = (x["q"], x["k"], x["v"], x["do"], x["gq"], x["gk"], x["gv"], w.causal, w.scale)
    fb = (x["q"], x["k"], x["v"])
    ref = {}
    if len(rows):
        ref["gradq"], ref["graddo"] = oracle.bob_rows(*args, rows)
        ref["o"], ref["lse"] = oracle.forward_rows(*fb, w.causal, w.scale, rows)
        ref["dq"] = oracle.backward_rows(*fb, x["do"], w.causal, w.scale, rows)
    if len(cols):
        ref["gradk"], ref["gradv"] = oracle.bob_cols(*args, cols)
        ref["dk"], ref["dv"] = oracle.backward_cols(*fb, x["do"], w.causal, w.scale, cols)
    return ref


def gpu_sample(gpu: dict, b: int, h: int, rows, cols):
    got = {}
    for k in ("gradq", "graddo", "o", "dq", "lse"):
        if len(rows):
            got[k] = to64(gpu[k][b, h])[rows]
    for k in ("gradk", "gradv", "dk", "dv"):
        if len(cols):
            got[k] = to64(gpu[k][b, h])[cols]
    return got


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = set([0, N - 1, N // 2])
    rows |= set(rng.integers(0, N, size=count).tolist())
    return np.array(sorted(rows))


def make(w: Workload, seed: int = 0):
    return make_inputs(w, seed=seed, device="cpu")
