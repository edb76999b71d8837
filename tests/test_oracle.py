"""Pins for the fp64 oracle, checked against things other than itself.

The FlashBoB pages print no worked example, so every pin comes from the
mathematics of the object the FlashBoB abstract names (exact BoB of softmax
attention):

* brute-force Python loops for the forward (definition of softmax attention);
* central finite differences: the first backward against the forward, and
  BoB against the first backward, at N <= 8, d <= 4;
* exact symbolic differentiation (sympy) of a 3-token case;
* fp64 torch autograd double-backward with an explicit -inf causal mask;
* exact invariants that hold at any size (Euler homogeneity in dO and V,
  the Q -> aQ, K -> K/a symmetry, translation invariance in K and V);
* closed forms: causal row 0 and the one-token sequence.

A plausible slip anywhere in the oracle (a dropped adjoint term, a sign, a
transposed operand, a wrong mask) moves at least the finite-difference and
autograd pins.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rnd(seed, n, d, count, scale=1.0):
    rng = np.random.default_rng(seed)
    return [scale * rng.standard_normal((n, d)) for _ in range(count)]


def inner(a, b):
    return float(np.sum(a * b))


def first_backward_objective(q, k, v, do, gq, gk, gv, causal, scale):
    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
    return inner(gq, dq) + inner(gk, dk) + inner(gv, dv)


def central_difference(fn, arrays, which, h):
    """Gradient of fn(*arrays) with respect to arrays[which]."""
    base = [a.copy() for a in arrays]
    x = base[which]
    g = np.zeros_like(x)
    for idx in itertools.product(*(range(s) for s in x.shape)):
        old = x[idx]
        x[idx] = old + h
        fp = fn(*base)
        x[idx] = old - h
        fm = fn(*base)
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- forward ---

@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_brute_force_loops(causal):
    n, d, scale = 6, 3, 0.7
    q, k, v = rnd(1, n, d, 3)
    o, lse = oracle.forward(q, k, v, causal, scale)
    for i in range(n):
        keys = range(i + 1) if causal else range(n)
        z = sum(math.exp(scale * sum(q[i, t] * k[j, t] for t in range(d)))
                for j in keys)
        assert abs(lse[i] - math.log(z)) < 1e-12
        for t in range(d):
            num = sum(math.exp(scale * sum(q[i, u] * k[j, u] for u in range(d)))
                      * v[j, t] for j in keys)
            assert abs(o[i, t] - num / z) < 1e-12


def test_forward_row_blocking_is_exact():
    q, k, v = rnd(2, 37, 5, 3)
    o1, l1 = oracle.forward(q, k, v, True, 0.4, row_block=1)
    o2, l2 = oracle.forward(q, k, v, True, 0.4, row_block=37)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


# ---------------------------------------------------------- first backward ---

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    n, d, scale = 5, 3, 0.8
    q, k, v, do = rnd(3, n, d, 4)

    def f(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, causal, scale)
        return inner(do, o)

    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
    for which, analytic in enumerate((dq, dk, dv)):
        fd = central_difference(f, [q, k, v], which, 1e-6)
        assert rel_err(analytic, fd) < 1e-7, which


# ------------------------------------------------------------------- BoB ---

@pytest.mark.parametrize("causal,n,d", [(False, 4, 2), (True, 4, 2),
                                        (False, 7, 3), (True, 8, 4)])
def test_bob_matches_finite_differences(causal, n, d):
    """T1: central differences of L = <gQ,dQ>+<gK,dK>+<gV,dV>."""
    scale = 1.0 / math.sqrt(d) * 1.3
    q, k, v, do, gq, gk, gv = rnd(10 + n, n, d, 7)
    grads = oracle.bob(q, k, v, do, gq, gk, gv, causal, scale)
    names = ("gradQ", "gradK", "gradV", "graddO")
    # arrays[which] for which = 0 (Q), 1 (K), 2 (V), 3 (dO)
    fn = lambda q_, k_, v_, do_: first_backward_objective(  # noqa: E731
        q_, k_, v_, do_, gq, gk, gv, causal, scale)
    for which, name in enumerate(names):
        fd = central_difference(fn, [q, k, v, do], which, 1e-6)
        assert rel_err(grads[which], fd) < 1e-7, name


def torch_double_backward(q, k, v, do, gq, gk, gv, causal, scale):
    """BoB through torch fp64 autograd of a plain dense attention with an
    explicit -inf mask (a library route independent of the oracle)."""
    t = lambda a: torch.tensor(a, dtype=torch.float64,  # noqa: E731
                               requires_grad=True)
    Q, K, V, dO = t(q), t(k), t(v), t(do)
    S = scale * (Q @ K.T)
    if causal:
        n = S.shape[0]
        mask = torch.ones(n, n, dtype=torch.bool).triu(1)
        S = S.masked_fill(mask, float("-inf"))
    O = torch.softmax(S, dim=-1) @ V
    dQ, dK, dV = torch.autograd.grad(O, (Q, K, V), grad_outputs=dO,
                                     create_graph=True)
    L = ((torch.tensor(gq) * dQ).sum() + (torch.tensor(gk) * dK).sum()
         + (torch.tensor(gv) * dV).sum())
    return [x.detach().numpy() for x in torch.autograd.grad(L, (Q, K, V, dO))]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (17, 8), (64, 16)])
def test_bob_matches_torch_double_backward(causal, n, d):
    """T2: fp64 autograd double-backward (explicit -inf causal mask)."""
    scale = 0.3
    ins = rnd(100 + n, n, d, 7)
    ref = torch_double_backward(*ins, causal, scale)
    got = oracle.bob(*ins, causal, scale)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


@pytest.mark.parametrize("causal", [False, True])
def test_bob_matches_symbolic_differentiation(causal):
    """Exact derivative (sympy) of a 3-token, d=2 case.

    The test derives dQ, dK, dV itself by differentiating <dO, O>
    symbolically, forms L, and differentiates again: no formula is shared
    with the oracle.
    """
    sp = pytest.importorskip("sympy")
    n, d = 3, 2
    scale = sp.Rational(1, 2)
    syms = {name: sp.Matrix(n, d, lambda i, j, nm=name: sp.Symbol(f"{nm}{i}{j}"))
            for name in ("q", "k", "v", "do")}
    q, k, v, do = (syms[x] for x in ("q", "k", "v", "do"))
    rng = np.random.default_rng(7)
    vals = {name: rng.integers(-3, 4, size=(n, d)) / 4 for name in syms}
    cot = {name: rng.integers(-3, 4, size=(n, d)) / 4 for name in ("gq", "gk",
                                                                   "gv")}
    o = sp.zeros(n, d)
    for i in range(n):
        keys = range(i + 1) if causal else range(n)
        w = [sp.exp(scale * sum(q[i, t] * k[j, t] for t in range(d)))
             for j in keys]
        z = sum(w)
        for t in range(d):
            o[i, t] = sum(wj * v[j, t] for wj, j in zip(w, keys)) / z
    f = sum(do[i, t] * o[i, t] for i in range(n) for t in range(d))
    first = {name: sp.Matrix(n, d, lambda i, t, m=syms[name]: sp.diff(f, m[i, t]))
             for name in ("q", "k", "v")}
    L = sum(cot["g" + name][i, t] * first[name][i, t]
            for name in ("q", "k", "v") for i in range(n) for t in range(d))
    subs = {syms[name][i, t]: sp.Rational(int(vals[name][i, t] * 4), 4)
            for name in syms for i in range(n) for t in range(d)}
    got = oracle.bob(vals["q"], vals["k"], vals["v"], vals["do"], cot["gq"],
                     cot["gk"], cot["gv"], causal, 0.5)
    for out, name in zip(got, ("q", "k", "v", "do")):
        for i in range(n):
            for t in range(d):
                exact = float(sp.diff(L, syms[name][i, t]).subs(subs).evalf(30))
                assert abs(out[i, t] - exact) < 1e-12, (name, i, t)


# ------------------------------------------------------------- invariants ---

def _invariants(q, k, v, do, gq, gk, gv, gradq, gradk, gradv, graddo, causal,
                scale):
    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
    L = inner(gq, dq) + inner(gk, dk) + inner(gv, dv)
    i1 = inner(graddo, do) - L                                   # Euler in dO
    i2 = inner(gradv, v) - (inner(gq, dq) + inner(gk, dk))       # Euler in V
    i3 = (inner(gradq, q) - inner(gradk, k)) - (inner(gk, dk) - inner(gq, dq))
    i4k = np.max(np.abs(gradk.sum(axis=0)))                      # K shift
    i4v = np.max(np.abs(gradv.sum(axis=0)))                      # V shift
    return i1, i2, i3, i4k, i4v


@pytest.mark.parametrize("causal", [False, True])
def test_bob_exact_invariants(causal):
    """I1-I4: hold exactly for the true BoB at any size."""
    n, d, scale = 96, 8, 0.35
    ins = rnd(5, n, d, 7)
    outs = oracle.bob(*ins, causal, scale, row_block=32)
    for r in _invariants(*ins, *outs, causal, scale):
        assert abs(r) < 1e-10


def test_bob_linearity():
    """I5: gradQ/K/V linear in dO, graddO independent of dO, all four
    jointly linear in (gQ, gK, gV)."""
    n, d, scale = 20, 4, 0.6
    q, k, v, do, gq, gk, gv = rnd(6, n, d, 7)
    do2, gq2, gk2, gv2 = rnd(8, n, d, 4)
    a, b = 0.7, -1.9
    base = oracle.bob(q, k, v, do, gq, gk, gv, True, scale)
    other = oracle.bob(q, k, v, do2, gq, gk, gv, True, scale)
    mixed = oracle.bob(q, k, v, a * do + b * do2, gq, gk, gv, True, scale)
    for i in range(3):
        assert np.allclose(mixed[i], a * base[i] + b * other[i], atol=1e-11)
    assert np.allclose(mixed[3], base[3], atol=1e-12)
    c1 = oracle.bob(q, k, v, do, gq2, gk2, gv2, True, scale)
    c2 = oracle.bob(q, k, v, do, a * gq + b * gq2, a * gk + b * gk2,
                    a * gv + b * gv2, True, scale)
    for i in range(4):
        assert np.allclose(c2[i], a * base[i] + b * c1[i], atol=1e-11)


# ------------------------------------------------------------ closed forms ---

def test_bob_causal_row0_closed_form():
    """Row 0 under a causal mask sees one key: softmax is constant there, so
    gradQ_0 = 0 and graddO_0 = gV_0."""
    ins = rnd(9, 12, 5, 7)
    gradq, _, _, graddo = oracle.bob(*ins, True, 0.5)
    assert np.max(np.abs(gradq[0])) < 1e-14
    assert np.max(np.abs(graddo[0] - ins[6][0])) < 1e-14


def test_bob_single_token_closed_form():
    """N = 1: gradQ = gradK = gradV = 0 and graddO = gV."""
    ins = rnd(11, 1, 6, 7)
    for causal in (False, True):
        gradq, gradk, gradv, graddo = oracle.bob(*ins, causal, 0.9)
        assert np.max(np.abs(np.concatenate([gradq, gradk, gradv]))) < 1e-15
        assert np.max(np.abs(graddo - ins[6])) < 1e-15


def test_causal_equals_nonzero_block_of_lower_triangle():
    """Causal BoB on rows [0, m) equals causal BoB of the length-m prefix
    for the row-local outputs (row i never sees keys beyond i)."""
    n, m, d, scale = 30, 13, 4, 0.5
    ins = rnd(12, n, d, 7)
    full = oracle.bob(*ins, True, scale)
    pref = oracle.bob(*(x[:m] for x in ins), True, scale)
    assert np.max(np.abs(full[0][:m] - pref[0])) < 1e-13
    assert np.max(np.abs(full[3][:m] - pref[3])) < 1e-13


# ------------------------------------------------- blocking and sampling ---

@pytest.mark.parametrize("causal", [False, True])
def test_bob_row_blocking_and_sampling_agree(causal):
    n, d, scale = 45, 6, 0.4
    ins = rnd(13, n, d, 7)
    ref = oracle.bob(*ins, causal, scale, row_block=n)
    for rb in (1, 7, 16):
        got = oracle.bob(*ins, causal, scale, row_block=rb)
        for a, b in zip(got, ref):
            assert np.max(np.abs(a - b)) < 1e-12
    rows = np.array([0, 3, 44, 20])
    gq_r, gdo_r = oracle.bob_rows(*ins, causal, scale, rows, row_block=3)
    assert np.max(np.abs(gq_r - ref[0][rows])) < 1e-12
    assert np.max(np.abs(gdo_r - ref[3][rows])) < 1e-12
    cols = np.array([40, 44, 31])
    gk_c, gv_c = oracle.bob_cols(*ins, causal, scale, cols, row_block=5)
    assert np.max(np.abs(gk_c - ref[1][cols])) < 1e-12
    assert np.max(np.abs(gv_c - ref[2][cols])) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_forward_backward_sampling_agrees_with_full(causal):
    """The sampled forward / first-backward oracles (rows of O, LSE, dQ;
    columns of dK, dV) reproduce the full ones, whose own pins are the
    brute-force loops and finite differences above."""
    n, d, scale = 41, 5, 0.6
    q, k, v, do = rnd(21, n, d, 4)
    o, lse = oracle.forward(q, k, v, causal, scale)
    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
    rows = np.array([0, 1, 17, 40])
    o_r, lse_r = oracle.forward_rows(q, k, v, causal, scale, rows)
    assert np.max(np.abs(o_r - o[rows])) < 1e-12
    assert np.max(np.abs(lse_r - lse[rows])) < 1e-12
    assert np.max(np.abs(oracle.backward_rows(q, k, v, do, causal, scale, rows) - dq[rows])) < 1e-12
    cols = np.array([39, 2, 40, 23])
    dk_c, dv_c = oracle.backward_cols(q, k, v, do, causal, scale, cols, row_block=6)
    assert np.max(np.abs(dk_c - dk[cols])) < 1e-12
    assert np.max(np.abs(dv_c - dv[cols])) < 1e-12


def test_batched_wrappers_match_per_head():
    B, H, n, d = 2, 3, 9, 4
    rng = np.random.default_rng(14)
    ins = [rng.standard_normal((B, H, n, d)) for _ in range(7)]
    outs = oracle.bob_batched(*ins, True, 0.5)
    o, lse = oracle.forward_batched(*ins[:3], True, 0.5)
    grads = oracle.backward_batched(*ins[:4], True, 0.5)
    for b in range(B):
        for h in range(H):
            per = oracle.bob(*(x[b, h] for x in ins), True, 0.5)
            for a, c in zip(outs, per):
                assert np.max(np.abs(a[b, h] - c)) < 1e-13
            o1, l1 = oracle.forward(*(x[b, h] for x in ins[:3]), True, 0.5)
            assert np.max(np.abs(o[b, h] - o1)) < 1e-13
            assert np.max(np.abs(lse[b, h] - l1)) < 1e-13
            g1 = oracle.backward(*(x[b, h] for x in ins[:4]), True, 0.5)
            for a, c in zip(grads, g1):
                assert np.max(np.abs(a[b, h] - c)) < 1e-13
