"""ctypes binding to libfbob.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor metadata, allocates outputs and workspace with PyTorch (device
memory is PyTorch's job here), passes raw pointers and the current CUDA
stream, and turns status codes into exceptions.  If the library is missing it
raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

OP_FORWARD, OP_BACKWARD, OP_BOB = 0, 1, 2
PATH_SIMT, PATH_TCGEN05 = 0, 1
DTYPES = {torch.bfloat16: 0, torch.float32: 1}

STATUS = {
    0: "FBOB_OK",
    1: "FBOB_ERR_INVALID_ARG",
    2: "FBOB_ERR_UNSUPPORTED",
    3: "FBOB_ERR_WORKSPACE",
    4: "FBOB_ERR_CUDA",
    5: "FBOB_ERR_TIMEOUT",
}


class FbobError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("dtype", ctypes.c_int),
                ("causal", ctypes.c_int), ("scale", ctypes.c_float)]


_LIB = None
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_SHP = ctypes.POINTER(Shape)

_SIGNATURES = {
    "fbob_version": (ctypes.c_int, []),
    "fbob_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "fbob_workspace_size": (_SZ, [ctypes.c_int, _SHP]),
    "fbob_forward": (ctypes.c_int, [_SHP, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "fbob_backward": (ctypes.c_int,
                      [_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "fbob_bob": (ctypes.c_int, [_SHP] + [_P] * 14 + [_SZ, _P]),
    "fbob_status": (ctypes.c_int, [_P, _P]),
    "fbob_path": (ctypes.c_int, [ctypes.c_int, _SHP]),
    "fbob_force_path": (ctypes.c_int, [ctypes.c_int]),
    "fbob_set_profile_events": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int]),
    "fbob_last_launch_count": (ctypes.c_int, []),
    "fbob_selftest_wait_timeout": (ctypes.c_int, [_P, _SZ, ctypes.c_int, _P]),
    "fbob_bob_noalloc": (ctypes.c_int, [_SHP] + [_P] * 13 + [_P]),
    "fbob_noalloc_status": (ctypes.c_int, [_P]),
    "fbob_set_wait_limit": (ctypes.c_longlong, [ctypes.c_longlong]),
}


def library_path() -> str:
    return os.environ.get("FBOB_LIBRARY", LIB_PATH)


def lib():
    """Load libfbob.so (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(code: int, what: str):
    if code != 0:
        raise FbobError(code, what)


def make_shape(B, H, N, d, dtype, causal, scale) -> Shape:
    if dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {dtype}; use bfloat16 or float32")
    return Shape(int(B), int(H), int(N), int(d), DTYPES[dtype], int(bool(causal)),
                 float(scale))


def shape_of(x: torch.Tensor, causal: bool, scale: float | None) -> Shape:
    if x.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    B, H, N, d = x.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return make_shape(B, H, N, d, x.dtype, causal, scale)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensors(ref: torch.Tensor, named: dict, scalar_names=()):
    if not ref.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    for name, t in named.items():
        if t is None:  # an optional argument left out
            continue
        if t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, expected {ref.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if name in scalar_names:
            if t.dtype != torch.float32 or tuple(t.shape) != tuple(ref.shape[:3]):
                raise ValueError(f"{name} must be float32 {tuple(ref.shape[:3])}")
        elif t.dtype != ref.dtype or t.shape != ref.shape:
            raise ValueError(f"{name} must match q: {ref.dtype} {tuple(ref.shape)}")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_size(op: int, shape: Shape) -> int:
    n = lib().fbob_workspace_size(op, ctypes.byref(shape))
    if n == 0:
        raise FbobError(2, "fbob_workspace_size")
    return int(n)


def alloc_workspace(op: int, shape: Shape, device) -> torch.Tensor:
    return torch.empty(workspace_size(op, shape), dtype=torch.uint8, device=device)


def path(op: int, shape: Shape) -> int:
    return int(lib().fbob_path(op, ctypes.byref(shape)))


def force_path(p: int) -> int:
    """-1 = automatic, 0 = CUDA cores, 1 = tensor cores.  Returns the old
    setting."""
    return int(lib().fbob_force_path(int(p)))


def last_launch_count() -> int:
    return int(lib().fbob_last_launch_count())


def set_profile_events(events) -> None:
    arr = (_P * max(1, len(events)))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().fbob_set_profile_events(arr, len(events)), "fbob_set_profile_events")


def status(workspace: torch.Tensor) -> int:
    return int(lib().fbob_status(_ptr(workspace), _stream(workspace.device)))


def forward(q, k, v, causal: bool = False, scale: float | None = None,
            out=None, workspace=None):
    """Attention forward: returns (O, LSE)."""
    _check_tensors(q, {"k": k, "v": v})
    shp = shape_of(q, causal, scale)
    o, lse = out if out is not None else (
        torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32,
                                         device=q.device))
    ws = workspace if workspace is not None else alloc_workspace(OP_FORWARD, shp, q.device)
    _check(lib().fbob_forward(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                              _ptr(lse), _ptr(ws), ws.numel(), _stream(q.device)),
           "fbob_forward")
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False,
             scale: float | None = None, out=None, workspace=None):
    """First backward: returns (dQ, dK, dV)."""
    _check_tensors(q, {"k": k, "v": v, "o": o, "do": do, "lse": lse}, ("lse",))
    shp = shape_of(q, causal, scale)
    dq, dk, dv = out if out is not None else tuple(torch.empty_like(q) for _ in range(3))
    ws = workspace if workspace is not None else alloc_workspace(OP_BACKWARD, shp, q.device)
    _check(lib().fbob_backward(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                               _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(ws), ws.numel(), _stream(q.device)),
           "fbob_backward")
    return dq, dk, dv


def bob(q, k, v, o, lse, do, gq, gk, gv, causal: bool = False,
        scale: float | None = None, out=None, workspace=None):
    """Backward-over-backward: returns (gradQ, gradK, gradV, graddO), the
    gradient of <gQ,dQ> + <gK,dK> + <gV,dV> w.r.t. (Q, K, V, dO).  Any of gq,
    gk, gv may be None: a zero cotangent, whose work the kernels skip."""
    _check_tensors(q, {"k": k, "v": v, "o": o, "do": do, "gq": gq, "gk": gk,
                       "gv": gv, "lse": lse}, ("lse",))
    shp = shape_of(q, causal, scale)
    outs = out if out is not None else tuple(torch.empty_like(q) for _ in range(4))
    ws = workspace if workspace is not None else alloc_workspace(OP_BOB, shp, q.device)
    _check(lib().fbob_bob(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                          _ptr(lse), _ptr(do), _ptr(gq), _ptr(gk), _ptr(gv),
                          *(_ptr(t) for t in outs), _ptr(ws), ws.numel(),
                          _stream(q.device)),
           "fbob_bob")
    return tuple(outs)


def bob_noalloc(q, k, v, o, lse, do, gq, gk, gv, causal: bool = False,
                scale: float | None = None, out=None):
    """BoB through fbob_bob_noalloc: same results as ``bob``, for callers that
    cannot allocate device memory; the scratch comes from the library's
    fixed device array (outputs are allocated here only when ``out`` is
    None)."""
    _check_tensors(q, {"k": k, "v": v, "o": o, "do": do, "gq": gq, "gk": gk,
                       "gv": gv, "lse": lse}, ("lse",))
    shp = shape_of(q, causal, scale)
    outs = out if out is not None else tuple(torch.empty_like(q) for _ in range(4))
    _check(lib().fbob_bob_noalloc(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                  _ptr(lse), _ptr(do), _ptr(gq), _ptr(gk), _ptr(gv),
                                  *(_ptr(t) for t in outs), _stream(q.device)),
           "fbob_bob_noalloc")
    return tuple(outs)


def set_wait_limit(ns: int) -> int:
    """Limit of one device-side bounded wait in nanoseconds (0 = the 2 s
    default).  Returns the previous limit."""
    old = int(lib().fbob_set_wait_limit(int(ns)))
    if old < 0:
        raise ValueError(f"wait limit {ns} ns is out of range")
    return old


def noalloc_status(device=None) -> int:
    """Device-side status of the last ``bob_noalloc`` call on ``device``
    (synchronises that device's current stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return int(lib().fbob_noalloc_status(_stream(dev)))


def selftest_wait_timeout(workspace: torch.Tensor, limit_us: int) -> int:
    """Runs the bounded-wait self-test and returns the resulting status."""
    _check(lib().fbob_selftest_wait_timeout(_ptr(workspace), workspace.numel(),
                                            int(limit_us), _stream(workspace.device)),
           "fbob_selftest_wait_timeout")
    return status(workspace)
