"""Seeded synthetic attention workloads.

This module only draws random tensors; it holds none of the attention
arithmetic, so both the CUDA path's tests and the fp64 oracle can consume
the same inputs without sharing any computation.

The five workloads are the attention shapes FlashBoB is exercised on: a small
fp32 case, and bf16 causal cases from N=4096 up to N=262144 (the longest
sequence the FlashBoB abstract reports on one GPU).  The paper states no
batch, head count, head dimension or value distribution; those below are this
library's choice.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "INPUT_ORDER"]

#: order in which tensors are drawn from the generator
INPUT_ORDER = ("q", "k", "v", "do", "gq", "gk", "gv")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "fp32" or "bf16"
    causal: bool
    qk_std: float       # std of Q and K
    v_std: float        # std of V
    cot_std: float      # std of dO, gQ, gK, gV

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("fp32_n256_d64", 1, 1, 256, 64, "fp32", False, 1.0, 1.0, 1.0),
        Workload("bf16_causal_h8_n4096_d64", 1, 8, 4096, 64, "bf16", True,
                 1.0, 1.0, 0.1),
        Workload("bf16_causal_b2h16_n16384_d128", 2, 16, 16384, 128, "bf16",
                 True, 1.0, 1.0, 0.1),
        Workload("bf16_causal_peaked_h8_n65536_d128", 1, 8, 65536, 128, "bf16",
                 True, 1.5, 0.1, 0.1),
        Workload("bf16_causal_h4_n262144_d64", 1, 4, 262144, 64, "bf16", True,
                 1.0, 1.0, 0.1),
        # without the causal mask, at the length where dense BoB is stated
        # to fail and at the two longest lengths
        Workload("bf16_h4_n16384_d128", 1, 4, 16384, 128, "bf16", False,
                 1.0, 1.0, 0.1),
        Workload("bf16_h8_n65536_d128", 1, 8, 65536, 128, "bf16", False,
                 1.0, 1.0, 0.1),
        Workload("bf16_h4_n262144_d64", 1, 4, 262144, 64, "bf16", False,
                 1.0, 1.0, 0.1),
        # B*H = 3 with 256 blocks per head: the kernels take heads in groups
        # of two, so the last group is partial
        Workload("bf16_causal_b3_n32768_d128", 3, 1, 32768, 128, "bf16", True,
                 1.0, 1.0, 0.1),
        Workload("bf16_causal_b3_n32768_d64", 3, 1, 32768, 64, "bf16", True,
                 1.0, 1.0, 0.1),
        # profiling-sized cases (inputs still larger than L2 in total)
        Workload("bf16_causal_h8_n8192_d128", 1, 8, 8192, 128, "bf16", True,
                 1.0, 1.0, 0.1),
        Workload("bf16_causal_h16_n8192_d64", 1, 16, 8192, 64, "bf16", True,
                 1.0, 1.0, 0.1),
    )
}


def make_inputs(w: Workload, seed: int = 0, device="cpu"):
    """Draw Q, K, V, dO, gQ, gK, gV ~ N(0, std^2) from a CPU generator seeded
    with ``seed`` (in INPUT_ORDER), round to the workload dtype, and move them
    to ``device``.  Returns a dict of [B, H, N, d] contiguous tensors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (w.B, w.H, w.N, w.d)
    stds = {"q": w.qk_std, "k": w.qk_std, "v": w.v_std, "do": w.cot_std,
            "gq": w.cot_std, "gk": w.cot_std, "gv": w.cot_std}
    out = {}
    for name in INPUT_ORDER:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if stds[name] != 1.0:
            x.mul_(stds[name])
        out[name] = x.to(w.torch_dtype).to(device).contiguous()
    return out
