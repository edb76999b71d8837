"""The oracle's pins must catch plausible mistakes.

Each case plants one slip (a dropped adjoint term, a sign, a wrong operand,
a missing scale or mask) in a private copy of the oracle's BoB row-block
routine, on the CPU, and checks that the finite-difference pin then fails.
The real oracle is never modified.
"""
import inspect
import math
import textwrap

import numpy as np
import pytest

import oracle
from oracle import attention_oracle as ao

from test_oracle import central_difference, first_backward_objective, rnd

MUTATIONS = {
    "drop O->P adjoint": ("b_p += b_o @ v.T", "pass"),
    "sign of D adjoint": ("b_dd = -np.sum(p * b_ds, axis=1, keepdims=True)",
                          "b_dd = np.sum(p * b_ds, axis=1, keepdims=True)"),
    "wrong operand in dQ adjoint": ("b_k = scale * (ds.T @ gq_r)",
                                    "b_k = scale * (ds.T @ q_r)"),
    "no softmax centring": (
        "b_s = p * (b_p - np.sum(p * b_p, axis=1, keepdims=True))",
        "b_s = p * b_p"),
    "missing scale on S adjoint": ("b_q += scale * (b_s @ k)",
                                   "b_q += (b_s @ k)"),
    "drop D->dO adjoint": ("b_do += b_dd * o", "pass"),
    "transposed dP in dO adjoint": ("b_do += b_dp @ v", "b_do += b_dp.T @ v"),
}


def mutated_row_block(old, new):
    src = textwrap.dedent(inspect.getsource(ao._bob_row_block))
    assert src.count(old) == 1, old
    ns = dict(vars(ao))
    exec(src.replace(old, new), ns)  # noqa: S102 - test-only source mutation
    return ns["_bob_row_block"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_finite_difference_pin_catches(name, monkeypatch):
    fn = mutated_row_block(*MUTATIONS[name])
    monkeypatch.setattr(ao, "_bob_row_block", fn)
    caught = False
    for causal in (False, True):
        n, d = 5, 3
        scale = 0.9 / math.sqrt(d)
        q, k, v, do, gq, gk, gv = rnd(31, n, d, 7)
        grads = oracle.bob(q, k, v, do, gq, gk, gv, causal, scale)
        f = lambda q_, k_, v_, do_: first_backward_objective(  # noqa: E731
            q_, k_, v_, do_, gq, gk, gv, causal, scale)
        for which in range(4):
            fd = central_difference(f, [q, k, v, do], which, 1e-6)
            err = np.max(np.abs(grads[which] - fd)) / np.max(np.abs(fd))
            caught |= err > 1e-4
    assert caught, f"mutation '{name}' escaped the finite-difference pin"
