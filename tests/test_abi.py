"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/fbob.h declares, sizes workspaces, picks kernel
families, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import exact_second_order_two_gb300 as fbob
from exact_second_order_two_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbob.build_library()
    return fbob.lib()


def declared_functions():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fbob_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("fbob_forward", "fbob_backward", "fbob_bob", "fbob_workspace_size",
              "fbob_status", "fbob_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert lib.fbob_version() >= 100
    for code in range(6):
        assert lib.fbob_strerror(code)
    assert lib.fbob_strerror(99) == b"unknown status"


def shape(**kw):
    base = dict(B=1, H=2, N=100, d=64, dtype=0, causal=1, scale=0.125)
    base.update(kw)
    return B.Shape(**base)


def test_workspace_sizes(lib):
    s = shape()
    rows = 1 * 2 * 100
    fwd = lib.fbob_workspace_size(0, ctypes.byref(s))
    bwd = lib.fbob_workspace_size(1, ctypes.byref(s))
    bob = lib.fbob_workspace_size(2, ctypes.byref(s))
    assert fwd >= 256
    assert bwd >= 256 + 4 * rows
    assert bob >= 256 + 3 * 4 * rows
    # never an N x N buffer: the workspace is linear in N
    s2 = shape(N=200)
    bob2 = lib.fbob_workspace_size(2, ctypes.byref(s2))
    assert bob2 <= 2 * bob + 4096
    assert lib.fbob_workspace_size(7, ctypes.byref(s)) == 0
    assert lib.fbob_workspace_size(2, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), 1), (dict(d=0), 1), (dict(B=-1), 1), (dict(causal=2), 1),
    (dict(dtype=5), 2), (dict(d=256), 2), (dict(B=300, H=300), 2),
    (dict(scale=0.0), 1),
])
def test_invalid_shapes_rejected(lib, kw, code):
    s = shape(**kw)
    assert lib.fbob_workspace_size(2, ctypes.byref(s)) == 0
    assert lib.fbob_path(2, ctypes.byref(s)) == -1
    ptrs = [ctypes.c_void_p(256)] * 12 + [None]   # graddO is null
    rc = lib.fbob_bob(ctypes.byref(s), *ptrs, ctypes.c_void_p(4096), 1 << 30, None)
    # the null graddO pointer or the shape is reported; never success
    assert rc in (1, code)


def test_null_and_misaligned_pointers_rejected(lib):
    s = shape()
    good = ctypes.c_void_p(1 << 20)
    args = [good] * 13
    args[3] = None
    assert lib.fbob_bob(ctypes.byref(s), *args, good, 1 << 30, None) == 1
    args = [good] * 13
    args[0] = ctypes.c_void_p((1 << 20) + 8)
    assert lib.fbob_bob(ctypes.byref(s), *args, good, 1 << 30, None) == 1
    assert lib.fbob_forward(None, good, good, good, good, good, good, 1 << 20, None) == 1


def test_null_cotangents_are_accepted_misaligned_ones_rejected(lib):
    """gq, gk, gv (arguments 6-8) may be NULL (zero cotangents); a present
    one must still be 16-byte aligned.  The workspace given is too small, so
    an accepted call stops at FBOB_ERR_WORKSPACE before touching a device."""
    s = shape()
    good = ctypes.c_void_p(1 << 20)
    for nulls in ((6,), (7,), (8,), (6, 7), (6, 8), (7, 8), (6, 7, 8)):
        args = [good] * 13
        for i in nulls:
            args[i] = None
        assert lib.fbob_bob(ctypes.byref(s), *args, good, 16, None) == 3, nulls
    args = [good] * 13
    args[6] = None
    args[7] = ctypes.c_void_p((1 << 20) + 8)
    assert lib.fbob_bob(ctypes.byref(s), *args, good, 16, None) == 1


def test_kernel_family_choice(lib):
    """bf16 at d = 64 / 128 takes the tcgen05 kernels for all three calls;
    fp32 and other head sizes take the CUDA-core kernels."""
    for op in (fbob.OP_FORWARD, fbob.OP_BACKWARD, fbob.OP_BOB):
        fp32 = shape(dtype=1)
        assert lib.fbob_path(op, ctypes.byref(fp32)) == fbob.PATH_SIMT
        odd = shape(d=40)
        assert lib.fbob_path(op, ctypes.byref(odd)) == fbob.PATH_SIMT
        for d in (64, 128):
            assert lib.fbob_path(op, ctypes.byref(shape(d=d))) == fbob.PATH_TCGEN05
    old = lib.fbob_force_path(0)
    try:
        for op in (fbob.OP_FORWARD, fbob.OP_BACKWARD, fbob.OP_BOB):
            assert lib.fbob_path(op, ctypes.byref(shape(d=128))) == fbob.PATH_SIMT
    finally:
        lib.fbob_force_path(old)


def test_workspace_sizes_per_family(lib):
    """The tcgen05 first backward and BoB need the fp32 dQ / gradQ accumulator
    (B*H*N*d*4 bytes) on top of the row scalars; the forward needs only the
    status word."""
    s = shape(d=128)
    rows = s.B * s.H * s.N
    acc = rows * s.d * 4
    fwd = lib.fbob_workspace_size(fbob.OP_FORWARD, ctypes.byref(s))
    bwd = lib.fbob_workspace_size(fbob.OP_BACKWARD, ctypes.byref(s))
    bob = lib.fbob_workspace_size(fbob.OP_BOB, ctypes.byref(s))
    assert fwd == 256
    assert bwd >= 256 + rows * 4 + acc
    assert bob >= 256 + 3 * rows * 4 + acc


def test_profile_event_hook_validation(lib):
    assert lib.fbob_set_profile_events(None, -1) == 1
    assert lib.fbob_set_profile_events(None, 17) == 1
    assert lib.fbob_set_profile_events(None, 0) == 0


def test_wait_limit_setting(lib):
    old = lib.fbob_set_wait_limit(5000)        # 5 us
    assert old == 2_000_000_000                 # the 2 s default
    assert lib.fbob_set_wait_limit(-1) == -1    # out of range: unchanged
    assert lib.fbob_set_wait_limit(61_000_000_000) == -1
    assert lib.fbob_set_wait_limit(0) == 5000   # 0 restores the default
    assert lib.fbob_set_wait_limit(0) == 2_000_000_000


def test_selftest_rejects_bad_arguments(lib):
    assert lib.fbob_selftest_wait_timeout(None, 256, 10, None) == 1
    assert lib.fbob_selftest_wait_timeout(ctypes.c_void_p(1 << 20), 16, 10, None) == 1
    assert lib.fbob_selftest_wait_timeout(ctypes.c_void_p(1 << 20), 256, 0, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.setenv("FBOB_LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()
