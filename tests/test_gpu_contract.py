"""GPU checks of the C ABI contract: outputs fully overwritten and nothing
written outside them (canaries, in place of a memory sanitizer), error
codes, and the device-side bounded-wait failure path."""
import math

import pytest
import torch

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300.synthetic import Workload, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

GUARD = 4096  # elements of guard region after every output


def guarded(like: torch.Tensor, fill=float("nan")):
    """A NaN-filled output tensor followed by a guard region in one buffer."""
    buf = torch.full((like.numel() + GUARD,), fill, dtype=like.dtype, device=like.device)
    return buf, buf[: like.numel()].view(like.shape)


@pytest.mark.parametrize("d,dtype,N", [(64, torch.bfloat16, 200), (128, torch.bfloat16, 333),
                                       (64, torch.float32, 77), (128, torch.bfloat16, 4096)])
def test_outputs_fully_written_and_guards_intact(d, dtype, N):
    w = Workload("canary", 1, 3, N, d, "bf16" if dtype == torch.bfloat16 else "fp32",
                 True, 1.0, 1.0, 0.2)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=11).items()}
    q = ins["q"]
    o_buf, o = guarded(q)
    lse_buf, lse = guarded(torch.empty(q.shape[:3], dtype=torch.float32, device="cuda"))
    fbob.forward(q, ins["k"], ins["v"], True, w.scale, out=(o, lse))
    bufs = [guarded(q) for _ in range(4)]
    fbob.bob(q, ins["k"], ins["v"], o, lse, ins["do"], ins["gq"], ins["gk"], ins["gv"],
             True, w.scale, out=tuple(b[1] for b in bufs))
    gbufs = [guarded(q) for _ in range(3)]
    fbob.backward(q, ins["k"], ins["v"], o, lse, ins["do"], True, w.scale,
                  out=tuple(b[1] for b in gbufs))
    torch.cuda.synchronize()
    for buf, view in [(o_buf, o), (lse_buf, lse)] + bufs + gbufs:
        assert torch.isfinite(view.float()).all()
        assert torch.isnan(buf[view.numel():].float()).all()


def test_workspace_guard_and_status():
    w = Workload("ws", 1, 2, 300, 128, "bf16", True, 1.0, 1.0, 0.2)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=12).items()}
    shp = fbob.shape_of(ins["q"], True, w.scale)
    need = fbob.workspace_size(fbob.OP_BOB, shp)
    ws_buf = torch.full((need + 8192,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = ws_buf[:need]
    o, lse = fbob.forward(ins["q"], ins["k"], ins["v"], True, w.scale)
    fbob.bob(ins["q"], ins["k"], ins["v"], o, lse, ins["do"], ins["gq"], ins["gk"],
             ins["gv"], True, w.scale, workspace=ws)
    assert fbob.status(ws) == 0
    assert (ws_buf[need:] == 0x5A).all()


def test_workspace_too_small_is_rejected():
    w = Workload("ws", 1, 1, 64, 64, "bf16", True, 1.0, 1.0, 0.2)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=1).items()}
    o, lse = fbob.forward(ins["q"], ins["k"], ins["v"], True, w.scale)
    shp = fbob.shape_of(ins["q"], True, w.scale)
    small = torch.empty(fbob.workspace_size(fbob.OP_BOB, shp) - 256, dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(fbob.FbobError) as e:
        fbob.bob(ins["q"], ins["k"], ins["v"], o, lse, ins["do"], ins["gq"], ins["gk"],
                 ins["gv"], True, w.scale, workspace=small)
    assert e.value.code == 3


def test_unsupported_head_dim_is_rejected():
    q = torch.zeros(1, 1, 8, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fbob.FbobError) as e:
        fbob.forward(q, q, q, True, 1 / math.sqrt(256))
    assert e.value.code == 2


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert fbob.selftest_wait_timeout(ws, 2000) == 5  # FBOB_ERR_TIMEOUT
    # the context is still usable afterwards
    w = Workload("after", 1, 1, 64, 64, "bf16", True, 1.0, 1.0, 0.2)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=2).items()}
    o, lse = fbob.forward(ins["q"], ins["k"], ins["v"], True, w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("d", [128, 64])
def test_real_kernels_stop_cleanly_when_their_waits_run_out(d):
    """fbob_bob with a 1 ns wait limit: the first wait of each thread block
    that is not already complete runs out.  That block records
    FBOB_ERR_TIMEOUT, every role of it stops, waits for its own copies and
    MMAs in flight, frees its TMEM and exits; the call reports the timeout
    through fbob_status, the GPU context stays usable, and the next call,
    with the default limit, is correct."""
    w = Workload("abort", 1, 2, 300, d, "bf16", True, 1.0, 1.0, 0.3)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=13).items()}
    args = (ins["q"], ins["k"], ins["v"])
    o, lse = fbob.forward(*args, True, w.scale)
    cot = (ins["do"], ins["gq"], ins["gk"], ins["gv"])
    ws = fbob.alloc_workspace(fbob.OP_BOB, fbob.shape_of(ins["q"], True, w.scale), "cuda")
    ref = fbob.bob(*args, o, lse, *cot, True, w.scale, workspace=ws)
    assert fbob.status(ws) == 0
    old = fbob.set_wait_limit(1)
    try:
        fbob.bob(*args, o, lse, *cot, True, w.scale, workspace=ws)
        st = fbob.status(ws)
    finally:
        fbob.set_wait_limit(old)
    assert st == 5  # FBOB_ERR_TIMEOUT
    got = fbob.bob(*args, o, lse, *cot, True, w.scale, workspace=ws)
    assert fbob.status(ws) == 0
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        err = ((g.double() - r.double()).abs().max() / r.double().abs().max()).item()
        assert err <= 1e-2, err


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("op", ["forward", "backward"])
def test_attention_kernels_stop_cleanly_when_their_waits_run_out(op, d):
    """The same 1 ns wait limit on the forward and on the first backward
    (whose reduce warp hands dQ^T partials to TMA reduce-adds): the call
    reports FBOB_ERR_TIMEOUT, and the next call with the default limit
    matches the one before.  A wait only gives up once the global timer has
    moved past its limit, and that timer ticks coarsely, so the problem is
    long enough (16 key tiles per row block) that some wait outlasts a tick."""
    w = Workload("abort_" + op, 1, 2, 2048, d, "bf16", True, 1.0, 1.0, 0.3)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=17).items()}
    args = (ins["q"], ins["k"], ins["v"])
    shp = fbob.shape_of(ins["q"], True, w.scale)
    if op == "forward":
        ws = fbob.alloc_workspace(fbob.OP_FORWARD, shp, "cuda")
        call = lambda: fbob.forward(*args, True, w.scale, workspace=ws)
    else:
        o, lse = fbob.forward(*args, True, w.scale)
        ws = fbob.alloc_workspace(fbob.OP_BACKWARD, shp, "cuda")
        call = lambda: fbob.backward(*args, o, lse, ins["do"], True, w.scale, workspace=ws)
    ref = [t.clone() for t in call()]
    assert fbob.status(ws) == 0
    old = fbob.set_wait_limit(1)
    try:
        call()
        st = fbob.status(ws)
    finally:
        fbob.set_wait_limit(old)
    assert st == 5  # FBOB_ERR_TIMEOUT
    got = call()
    assert fbob.status(ws) == 0
    torch.cuda.synchronize()
    # dQ sums partials from many blocks in no fixed order: compare with a
    # tolerance rather than bit for bit
    for g, r in zip(got, ref):
        err = ((g.double() - r.double()).abs().max() / r.double().abs().max()).item()
        assert err <= 1e-2, err


def test_launch_count_is_reported():
    w = Workload("count", 1, 1, 128, 64, "bf16", True, 1.0, 1.0, 0.2)
    ins = {k: v.cuda() for k, v in make_inputs(w, seed=3).items()}
    o, lse = fbob.forward(ins["q"], ins["k"], ins["v"], True, w.scale)
    fbob.bob(ins["q"], ins["k"], ins["v"], o, lse, ins["do"], ins["gq"], ins["gk"],
             ins["gv"], True, w.scale)
    assert fbob.last_launch_count() >= 2
