"""fbob_bob_noalloc, the BoB call for callers that cannot allocate device
memory (hosts that hand a kernel only its input and output buffers, or code
that must not call cudaMalloc / cudaFree), must give the same results as
fbob_bob with a caller-owned workspace, on two calls in a row through the C
ABI.

This file sorts last so that a run stopping at the first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300 import _binding as B
from exact_second_order_two_gb300.synthetic import Workload, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

TOL = 2e-2  # max|err| / max|ref|, the bf16 tolerance of the parity tests


def rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).abs().max() / b.abs().max().clamp_min(1e-30)).item()


def run_noalloc(shape, ins, o, lse):
    outs = tuple(torch.full_like(ins["q"], float("nan")) for _ in range(4))
    rc = B.lib().fbob_bob_noalloc(
        ctypes.byref(shape), *(B._ptr(ins[n]) for n in ("q", "k", "v")), B._ptr(o),
        B._ptr(lse), *(B._ptr(ins[n]) for n in ("do", "gq", "gk", "gv")),
        *(B._ptr(t) for t in outs), B._stream(ins["q"].device))
    return rc, outs


def check_against_workspace_entry_point(w, seeds, tol):
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    shape = B.make_shape(w.B, w.H, w.N, w.d, dtype, w.causal, w.scale)
    need = B.lib().fbob_workspace_size(fbob.OP_BOB, ctypes.byref(shape))
    assert 0 < need <= (32 << 20)
    for seed in seeds:                          # calls in a row
        ins = {k: v.cuda() for k, v in make_inputs(w, seed=seed).items()}
        o, lse = fbob.forward(ins["q"], ins["k"], ins["v"], w.causal, w.scale)
        ref = fbob.bob(ins["q"], ins["k"], ins["v"], o, lse, ins["do"], ins["gq"],
                       ins["gk"], ins["gv"], w.causal, w.scale)
        rc, outs = run_noalloc(shape, ins, o, lse)
        assert rc == 0, B.STATUS.get(rc, rc)
        # the device-side status of that call (bounded waits) reads back clean
        assert fbob.noalloc_status() == 0
        torch.cuda.synchronize()
        for name, got, want in zip(("gradQ", "gradK", "gradV", "graddO"), outs, ref):
            assert torch.isfinite(got.float()).all(), name
            assert rel(got, want) <= tol, (name, seed, rel(got, want))
        del ins, o, lse, ref, outs


@pytest.mark.parametrize("d,N,heads", [(128, 700, 3), (64, 1000, 2)])
def test_noalloc_matches_workspace_entry_point_twice(d, N, heads):
    fbob.build_library()
    w = Workload("noalloc", 1, heads, N, d, "bf16", True, 1.0, 1.0, 0.3)
    check_against_workspace_entry_point(w, (21, 22), TOL)


def test_noalloc_on_cuda_cores_twice():
    """fp32 at d = 40 runs the CUDA-core kernels, whose scratch layout (row
    scalars only, no gradQ accumulator) differs from the tensor-core one."""
    fbob.build_library()
    w = Workload("noalloc_simt", 2, 1, 300, 40, "fp32", True, 1.0, 1.0, 0.3)
    check_against_workspace_entry_point(w, (23, 24), 1e-4)


def largest_n_that_fits(d):
    lo, hi = 1, 1 << 22
    limit = 32 << 20
    while lo < hi:                    # largest N with need <= limit
        mid = (lo + hi + 1) // 2
        s = B.make_shape(1, 1, mid, d, torch.bfloat16, True, d ** -0.5)
        need = B.lib().fbob_workspace_size(fbob.OP_BOB, ctypes.byref(s))
        if 0 < need <= limit:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_at_the_scratch_limit():
    """A problem whose workspace just fits uses the array up to its end and
    still matches; one row more is rejected with FBOB_ERR_WORKSPACE."""
    fbob.build_library()
    n = largest_n_that_fits(128)
    assert n > 60000
    w = Workload("noalloc_limit", 1, 1, n, 128, "bf16", True, 1.0, 1.0, 0.3)
    check_against_workspace_entry_point(w, (25, 26), TOL)
    q = torch.zeros(1, 1, n + 1, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, n + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(fbob.FbobError) as e:
        fbob.bob_noalloc(q, q, q, q, lse, q, q, q, q, True)
    assert e.value.code == 3   # FBOB_ERR_WORKSPACE


def test_noalloc_rejects_problems_beyond_its_scratch():
    fbob.build_library()
    q = torch.zeros(1, 4, 65536, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 4, 65536, dtype=torch.float32, device="cuda")
    with pytest.raises(fbob.FbobError) as e:
        fbob.bob_noalloc(q, q, q, q, lse, q, q, q, q, True)
    assert e.value.code == 3   # FBOB_ERR_WORKSPACE: needs more than 32 MiB
