"""Plain fp64 CPU oracle for softmax attention, its first backward, and the
exact backward-over-backward (BoB) that FlashBoB computes.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, constant or helper with the CUDA
library; the two meet only in the seeded input generator.

Source: "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
Attention", Abstract.  The abstract defines the object (exact BoB of softmax
attention: the gradient, with respect to the attention inputs, of a scalar
built from the first backward's outputs) but prints no equations.  The
oracle therefore does NOT use the paper's two-row-scalar factorisation at
all.  It writes out the plain definition instead:

  forward        S = c Q K^T (masked), LSE = logsumexp_row(S),
                 P = exp(S - LSE), O = P V
  first backward dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D),
                 dQ = c dS K, dK = c dS^T Q, dV = P^T dO
  BoB            the gradient of  L = <gQ,dQ> + <gK,dK> + <gV,dV>
                 with respect to (Q, K, V, dO), obtained by reverse-mode
                 differentiation of the first-backward lines above, one
                 adjoint line per forward line, in reverse order.

Readings taken where the pages are silent:
  * O and LSE are functions of Q, K, V (total derivative), not free inputs.
  * LSE is the natural log of the row sum of exp of the *scaled* scores.
  * causal masking is square and top-left aligned: key j is visible to query
    i iff j <= i.
  * the scale c is a constant argument and is not differentiated.

Every function works on one (batch, head) slice: arrays of shape [N, d] in
float64.  Batched helpers at the bottom loop over leading dimensions.
Large N is handled by processing query rows in blocks; the gradient of the
row-local quantities is exact per block, and the column-side gradients
(gradK, gradV) are sums over blocks.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "forward",
    "backward",
    "bob",
    "bob_rows",
    "bob_cols",
    "forward_batched",
    "backward_batched",
    "bob_batched",
    "default_row_block",
]


def default_row_block(n_keys: int, budget_bytes: int = 1 << 27) -> int:
    """Rows per block so that one [rows, n_keys] float64 matrix stays near
    ``budget_bytes``; purely a memory knob, it does not change any result."""
    return int(max(1, min(1024, budget_bytes // (8 * max(1, n_keys)))))


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _visible(rows: np.ndarray, n_keys: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_keys]: which keys each query row may attend to."""
    cols = np.arange(n_keys)
    if causal:
        return cols[None, :] <= rows[:, None]
    return np.ones((rows.size, n_keys), dtype=bool)


def _row_block_forward(q, k, v, rows, causal, scale):
    """Forward quantities for the query rows ``rows`` (full rows of P)."""
    n = k.shape[0]
    mask = _visible(rows, n, causal)
    s = scale * (q[rows] @ k.T)                      # S = c Q K^T
    s_masked = np.where(mask, s, -np.inf)
    m = np.max(s_masked, axis=1, keepdims=True)      # every row sees key 0
    lse = m + np.log(np.sum(np.exp(s_masked - m), axis=1, keepdims=True))
    p = np.where(mask, np.exp(s_masked - lse), 0.0)  # P = exp(S - LSE)
    o = p @ v                                        # O = P V
    return mask, p, o, lse[:, 0]


# --------------------------------------------------------------------------
# forward and first backward (what BoB differentiates)
# --------------------------------------------------------------------------

def forward(q, k, v, causal: bool, scale: float, row_block: int | None = None):
    """Softmax attention forward: returns (O [N,d], LSE [N]).

    FlashAttention's forward (cited by the FlashBoB abstract as the
    I/O-efficient forward BoB builds on): O = softmax(c Q K^T) V, with the
    row log-sum-exp kept for the backward passes.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    o = np.zeros((n, v.shape[1]))
    lse = np.zeros(n)
    for r0 in range(0, n, rb):
        rows = np.arange(r0, min(n, r0 + rb))
        _, _, o_blk, lse_blk = _row_block_forward(q, k, v, rows, causal, scale)
        o[rows] = o_blk
        lse[rows] = lse_blk
    return o, lse


def backward(q, k, v, do, causal: bool, scale: float,
             row_block: int | None = None):
    """First backward of softmax attention: returns (dQ, dK, dV).

    D_i = sum_k dO_ik O_ik;  dS = P * (dP - D);  dQ = c dS K;
    dK = c dS^T Q;  dV = P^T dO  (the "first backward pass" the FlashBoB
    abstract says FlashAttention already makes I/O-efficient).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, n, rb):
        rows = np.arange(r0, min(n, r0 + rb))
        _, p, o, _ = _row_block_forward(q, k, v, rows, causal, scale)
        dp = do[rows] @ v.T                               # dP = dO V^T
        dd = np.sum(do[rows] * o, axis=1, keepdims=True)  # D = rowsum(dO*O)
        ds = p * (dp - dd)                                # dS = P*(dP - D)
        dq[rows] = scale * (ds @ k)                       # dQ = c dS K
        dk += scale * (ds.T @ q[rows])                    # dK = c dS^T Q
        dv += p.T @ do[rows]                              # dV = P^T dO
    return dq, dk, dv


def forward_rows(q, k, v, causal: bool, scale: float, rows):
    """O and LSE at the query rows ``rows`` only (row-local, so large-N
    sampling costs O(len(rows) * N * d)); same definition as ``forward``."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    rows = np.asarray(rows, dtype=np.int64)
    _, _, o, lse = _row_block_forward(q, k, v, rows, causal, scale)
    return o, lse


def backward_rows(q, k, v, do, causal: bool, scale: float, rows):
    """dQ at the query rows ``rows`` only: row i of dS needs row i of P and
    D_i alone, so this is row-local; same definition as ``backward``."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    rows = np.asarray(rows, dtype=np.int64)
    _, p, o, _ = _row_block_forward(q, k, v, rows, causal, scale)
    dp = do[rows] @ v.T
    dd = np.sum(do[rows] * o, axis=1, keepdims=True)
    return scale * ((p * (dp - dd)) @ k)


def backward_cols(q, k, v, do, causal: bool, scale: float, cols,
                  row_block: int | None = None):
    """dK and dV at the key rows ``cols`` only: column j sums over every
    query row that sees key j (rows i >= min(cols) when causal); same
    definition as ``backward``."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    cols = np.asarray(cols, dtype=np.int64)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    first = int(cols.min()) if causal else 0
    dk = np.zeros((cols.size, k.shape[1]))
    dv = np.zeros((cols.size, v.shape[1]))
    for r0 in range(first, n, rb):
        rows = np.arange(r0, min(n, r0 + rb))
        _, p, o, _ = _row_block_forward(q, k, v, rows, causal, scale)
        dp = do[rows] @ v[cols].T
        dd = np.sum(do[rows] * o, axis=1, keepdims=True)
        ds = p[:, cols] * (dp - dd)
        dk += scale * (ds.T @ q[rows])
        dv += p[:, cols].T @ do[rows]
    return dk, dv


# --------------------------------------------------------------------------
# backward-over-backward
# --------------------------------------------------------------------------

def _bob_row_block(q, k, v, do, gq, gk, gv, rows, causal, scale):
    """Reverse-mode adjoint of the first backward restricted to query rows
    ``rows``.

    Returns the row-local results (gradQ[rows], graddO[rows]) and this
    block's contributions to the column-side results as full [N, d] arrays
    (gradK_part, gradV_part).  Each adjoint line below is the transpose of
    one line of ``backward`` (plus the forward it recomputes), taken in
    reverse order; ``b_X`` is the cotangent of X.
    """
    # ---- recompute the forward and the first backward for these rows ----
    _, p, o, _ = _row_block_forward(q, k, v, rows, causal, scale)
    q_r, gq_r, do_r = q[rows], gq[rows], do[rows]
    dp = do_r @ v.T                                   # dP = dO V^T
    dd = np.sum(do_r * o, axis=1, keepdims=True)      # D = rowsum(dO*O)
    ds = p * (dp - dd)                                # dS = P*(dP - D)

    # ---- seed: L = <gQ,dQ> + <gK,dK> + <gV,dV> ----
    # dV = P^T dO          ->  b_P += dO gV^T ;  b_dO += P gV
    b_p = do_r @ gv.T
    b_do = p @ gv
    # dK = c dS^T Q        ->  b_dS += c Q gK^T ;  b_Q += c dS gK
    b_ds = scale * (q_r @ gk.T)
    b_q = scale * (ds @ gk)
    # dQ = c dS K          ->  b_dS += c gQ K^T ;  b_K += c dS^T gQ
    b_ds += scale * (gq_r @ k.T)
    b_k = scale * (ds.T @ gq_r)
    b_v = np.zeros_like(v)

    # dS = P * (dP - D)    ->  b_P += b_dS*(dP - D); b_dP = P*b_dS;
    #                          b_D = -rowsum(P*b_dS)
    b_p += b_ds * (dp - dd)
    b_dp = p * b_ds
    b_dd = -np.sum(p * b_ds, axis=1, keepdims=True)
    # D = rowsum(dO * O)   ->  b_dO += b_D O ;  b_O = b_D dO
    b_do += b_dd * o
    b_o = b_dd * do_r
    # O = P V              ->  b_P += b_O V^T ;  b_V += P^T b_O
    b_p += b_o @ v.T
    b_v += p.T @ b_o
    # dP = dO V^T          ->  b_dO += b_dP V ;  b_V += b_dP^T dO
    b_do += b_dp @ v
    b_v += b_dp.T @ do_r
    # P = exp(S - logsumexp(S))  ->  b_S = P * (b_P - rowsum(P*b_P))
    b_s = p * (b_p - np.sum(p * b_p, axis=1, keepdims=True))
    # S = c Q K^T          ->  b_Q += c b_S K ;  b_K += c b_S^T Q
    b_q += scale * (b_s @ k)
    b_k += scale * (b_s.T @ q_r)
    return b_q, b_do, b_k, b_v


def _check_shapes(q, k, v, do, gq, gk, gv):
    n, d = q.shape
    for name, x in (("k", k), ("v", v), ("do", do), ("gq", gq), ("gk", gk),
                    ("gv", gv)):
        if x.shape != (n, d):
            raise ValueError(f"{name} has shape {x.shape}, expected {(n, d)}")


def bob(q, k, v, do, gq, gk, gv, causal: bool, scale: float,
        row_block: int | None = None):
    """Exact backward-over-backward of softmax attention.

    Returns (gradQ, gradK, gradV, graddO): the gradient of
    L = <gQ,dQ> + <gK,dK> + <gV,dV> with respect to Q, K, V and dO, where
    (dQ, dK, dV) is ``backward(q, k, v, do)``.  This is the quantity the
    FlashBoB abstract calls exact BoB of softmax attention.
    """
    q, k, v, do, gq, gk, gv = (_as64(x) for x in (q, k, v, do, gq, gk, gv))
    _check_shapes(q, k, v, do, gq, gk, gv)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    gradq = np.zeros_like(q)
    graddo = np.zeros_like(do)
    gradk = np.zeros_like(k)
    gradv = np.zeros_like(v)
    for r0 in range(0, n, rb):
        rows = np.arange(r0, min(n, r0 + rb))
        b_q, b_do, b_k, b_v = _bob_row_block(q, k, v, do, gq, gk, gv, rows,
                                             causal, scale)
        gradq[rows] = b_q
        graddo[rows] = b_do
        gradk += b_k
        gradv += b_v
    return gradq, gradk, gradv, graddo


def bob_rows(q, k, v, do, gq, gk, gv, causal: bool, scale: float, rows,
             row_block: int | None = None):
    """gradQ and graddO at the query rows ``rows`` only.

    Both are row-local (row i depends only on row i of P and the keys it
    sees), so this costs O(len(rows) * N * d) and serves large-N sampling.
    """
    q, k, v, do, gq, gk, gv = (_as64(x) for x in (q, k, v, do, gq, gk, gv))
    rows = np.asarray(rows, dtype=np.int64)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    gq_out = np.zeros((rows.size, q.shape[1]))
    gdo_out = np.zeros((rows.size, do.shape[1]))
    for b0 in range(0, rows.size, rb):
        sel = rows[b0:b0 + rb]
        b_q, b_do, _, _ = _bob_row_block(q, k, v, do, gq, gk, gv, sel, causal,
                                         scale)
        gq_out[b0:b0 + sel.size] = b_q
        gdo_out[b0:b0 + sel.size] = b_do
    return gq_out, gdo_out


def bob_cols(q, k, v, do, gq, gk, gv, causal: bool, scale: float, cols,
             row_block: int | None = None):
    """gradK and gradV at the key rows ``cols`` only.

    Column j collects contributions from every query row that sees key j
    (all rows, or rows i >= min(cols) when causal), each of which needs its
    full softmax row; so this costs O(#contributing rows * N * d).  Under a
    causal mask, columns near the end of the sequence are cheap.
    """
    q, k, v, do, gq, gk, gv = (_as64(x) for x in (q, k, v, do, gq, gk, gv))
    cols = np.asarray(cols, dtype=np.int64)
    n = q.shape[0]
    rb = row_block or default_row_block(n)
    first = int(cols.min()) if causal else 0
    gk_out = np.zeros((cols.size, k.shape[1]))
    gv_out = np.zeros((cols.size, v.shape[1]))
    for r0 in range(first, n, rb):
        rows = np.arange(r0, min(n, r0 + rb))
        _, _, b_k, b_v = _bob_row_block(q, k, v, do, gq, gk, gv, rows, causal,
                                        scale)
        gk_out += b_k[cols]
        gv_out += b_v[cols]
    return gk_out, gv_out


# --------------------------------------------------------------------------
# batched wrappers: arrays of shape [..., N, d]
# --------------------------------------------------------------------------

def _heads(x):
    x = _as64(x)
    return x.reshape((-1,) + x.shape[-2:]), x.shape[:-2]


def forward_batched(q, k, v, causal, scale, row_block=None):
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    outs = [forward(qh[h], kh[h], vh[h], causal, scale, row_block)
            for h in range(qh.shape[0])]
    o = np.stack([x[0] for x in outs]).reshape(lead + qh.shape[-2:])
    lse = np.stack([x[1] for x in outs]).reshape(lead + qh.shape[-2:-1])
    return o, lse


def backward_batched(q, k, v, do, causal, scale, row_block=None):
    hs = [_heads(x)[0] for x in (q, k, v, do)]
    lead = np.shape(q)[:-2]
    outs = [backward(*(x[h] for x in hs), causal, scale, row_block)
            for h in range(hs[0].shape[0])]
    return tuple(np.stack([o[i] for o in outs]).reshape(np.shape(q))
                 for i in range(3))


def bob_batched(q, k, v, do, gq, gk, gv, causal, scale, row_block=None):
    hs = [_heads(x)[0] for x in (q, k, v, do, gq, gk, gv)]
    outs = [bob(*(x[h] for x in hs), causal, scale, row_block)
            for h in range(hs[0].shape[0])]
    return tuple(np.stack([o[i] for o in outs]).reshape(np.shape(q))
                 for i in range(4))
