"""GB300-native FlashBoB: exact backward-over-backward of softmax attention.

The computation lives in libfbob.so (hand-written sm_103a CUDA behind a C
ABI, ``include/fbob.h``).  This package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    OP_BACKWARD,
    OP_BOB,
    OP_FORWARD,
    PATH_SIMT,
    PATH_TCGEN05,
    FbobError,
    Shape,
    alloc_workspace,
    backward,
    bob,
    bob_noalloc,
    force_path,
    forward,
    last_launch_count,
    lib,
    make_shape,
    noalloc_status,
    path,
    selftest_wait_timeout,
    set_profile_events,
    set_wait_limit,
    shape_of,
    status,
    workspace_size,
)
from .autograd import attention  # noqa: F401
from . import meta  # noqa: F401
from .build import build_library  # noqa: F401

__version__ = "0.1.0"
