"""fp64 reference attention: the plain definition, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This module is the
oracle the CUDA kernels are checked against; it never imports the product
package and the product never imports it.

Conventions (shared with the source pages' statement of the problem):

* Q, K, V, dO are arrays of shape [..., N, d] (in practice [B, H, N, d];
  [V1详解 §8.1]: the leading dims are batch and head and pass through, the
  last two dims are the matrix).  Every leading index is an independent
  attention problem.
* ``scale`` multiplies Q K^T; the pages use 1/sqrt(d) [V1详解 §1.1].
* ``causal``: key j is visible to query i iff j <= i (square, top-left
  aligned).  The pages name the causal mask but never define it
  [v1～v4 v4 §4]; this is the plainest reading.
* L is the natural-log logsumexp of each score row, L = m + log(l)
  [v1～v4 v2 §1].

All arithmetic is float64.  Inputs are widened exactly (bf16 and fp32 are
subsets of fp64), so the oracle's only error is fp64 rounding.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def to_f64(t) -> np.ndarray:
    """Widen a torch tensor (any float dtype, any device) or array to fp64.

    bf16 -> fp64 and fp32 -> fp64 are exact, so the oracle sees the very
    values the kernels see.
    """
    if isinstance(t, np.ndarray):
        return t.astype(np.float64, copy=False)
    import torch  # local import: plain CPU data movement only

    return t.detach().to(device="cpu", dtype=torch.float64).numpy()


def _heads(x: np.ndarray) -> tuple[np.ndarray, tuple]:
    """View [..., N, d] as [P, N, d] where P is the product of leading dims."""
    lead = x.shape[:-2]
    return x.reshape((-1,) + x.shape[-2:]), lead


def _visible_mask(rows: np.ndarray, n_k: int, causal: bool) -> np.ndarray | None:
    """Boolean [len(rows), n_k]: True where key j is visible to query rows[r]."""
    if not causal:
        return None
    cols = np.arange(n_k)
    return cols[None, :] <= rows[:, None]


def _scores(qh: np.ndarray, kh: np.ndarray, rows: np.ndarray, causal: bool,
            scale: float) -> np.ndarray:
    """S = scale * Q_rows K^T with masked entries set to -inf.

    [V1详解 §1.1] S = Q K^T / sqrt(d); the mask replaces hidden entries by
    -inf so that their softmax weight is exactly zero.
    """
    s = scale * (qh[rows] @ kh.T)
    vis = _visible_mask(rows, kh.shape[0], causal)
    if vis is not None:
        s = np.where(vis, s, NEG_INF)
    return s


def _softmax_rows(s: np.ndarray):
    """Safe softmax of each row of s, with its statistics.

    [V1详解 §3.1] (three passes): m = max, l = sum exp(x - m),
    y = exp(x - m) / l.  Returns (P, m, l, L) with L = m + log l
    [v1～v4 v2 §1].  A row with no visible entry (never produced by square
    causal attention) gets P = 0, m = -inf, l = 0, L = -inf.
    """
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l[:, None] > 0, e / l[:, None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(l), NEG_INF)
    return p, m, l, lse


# --------------------------------------------------------------------------
# softmax on a vector: three-pass and blockwise-online
# --------------------------------------------------------------------------

def softmax_three_pass(x) -> tuple[np.ndarray, float, float]:
    """Safe softmax of a 1-D vector by the three passes of [V1详解 §3.1].

    Returns (y, m, l): pass 1 takes m = max x, pass 2 l = sum exp(x - m),
    pass 3 y = exp(x - m) / l.
    """
    x = np.asarray(x, dtype=np.float64)
    m = -math.inf
    for xi in x:                      # pass 1
        m = max(m, float(xi))
    l = 0.0
    for xi in x:                      # pass 2
        l += math.exp(float(xi) - m)
    y = np.array([math.exp(float(xi) - m) / l for xi in x])   # pass 3
    return y, m, l


def online_softmax_blockwise(x, block: int):
    """Online softmax over consecutive blocks of a 1-D vector.

    [V1详解 §3.2] / [v1～v4 v1 §2]: keep a running max m and a sum l taken
    relative to m.  For each new block b:
        m_new = max(m, max b)
        l     = l * exp(m - m_new) + sum exp(b - m_new)
    and at the end y = exp(x - m) / l.  Returns (y, m, l, history) where
    history lists (m, l) after every block (the page's worked example quotes
    exactly these intermediate pairs).  m starts at -inf and l at 0; while m
    is still -inf the correction factor is taken as 1 (nothing has been
    accumulated yet, so its value does not matter).
    """
    x = np.asarray(x, dtype=np.float64)
    m, l = -math.inf, 0.0
    history = []
    for start in range(0, len(x), block):
        b = x[start:start + block]
        m_new = max(m, float(b.max()))
        if m_new == -math.inf:
            history.append((m, l))
            continue
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        l = l * alpha + float(np.exp(b - m_new).sum())
        m = m_new
        history.append((m, l))
    y = np.exp(x - m) / l
    return y, m, l, history


# --------------------------------------------------------------------------
# attention forward: the definition
# --------------------------------------------------------------------------

def _head_forward_rows(qh, kh, vh, rows, causal, scale):
    """O and L of the given query rows of one head, straight from the
    definition [V1详解 §1.1]: S = scale Q K^T, P = softmax(S), O = P V.

    For causal attention, the columns beyond the last visible key of these
    rows carry weight exactly 0 (exp(-inf)); they are left out of the
    product, which changes no value.
    """
    rows = np.asarray(rows)
    n_k = kh.shape[0]
    if causal and len(rows):
        n_k = min(n_k, int(rows.max()) + 1)
    s = _scores(qh, kh[:n_k], rows, causal, scale)
    p, _, _, lse = _softmax_rows(s)
    return p @ vh[:n_k], lse


def attention_forward(q, k, v, causal: bool, scale: float, row_chunk: int = 2048):
    """Exact attention forward.  Returns (O, L), O [..., N, d], L [..., N].

    [V1详解 §1.1]: S = Q K^T * scale, P = softmax(S) (row-wise), O = P V.
    [v1～v4 v2 §1]: L = m + log l per row.  Rows are evaluated in chunks of
    ``row_chunk`` (each row's value depends on that row only).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    n = qh.shape[1]
    o = np.empty(qh.shape[:2] + (vh.shape[2],))
    lse = np.empty(qh.shape[:2])
    for h in range(qh.shape[0]):
        for r0 in range(0, n, row_chunk):
            rows = np.arange(r0, min(n, r0 + row_chunk))
            o[h, rows], lse[h, rows] = _head_forward_rows(qh[h], kh[h], vh[h], rows,
                                                         causal, float(scale))
    return o.reshape(lead + o.shape[1:]), lse.reshape(lead + lse.shape[1:])


def attention_forward_rows(q, k, v, rows, causal: bool, scale: float):
    """O and L for selected query rows only.

    ``rows`` is either a 1-D index array (same rows in every head) or an
    array of shape [..., R] matching the leading dims of q.  Returns
    O [..., R, d] and L [..., R].  Same definition as attention_forward.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    rows = np.asarray(rows)
    per_head = rows.reshape(-1, rows.shape[-1]) if rows.ndim > 1 else None
    r = rows.shape[-1]
    o = np.empty((qh.shape[0], r, vh.shape[2]))
    lse = np.empty((qh.shape[0], r))
    for h in range(qh.shape[0]):
        rr = per_head[h] if per_head is not None else rows
        o[h], lse[h] = _head_forward_rows(qh[h], kh[h], vh[h], rr, causal, float(scale))
    return o.reshape(lead + o.shape[1:]), lse.reshape(lead + lse.shape[1:])


def attention_lse_all_rows(q, k, causal: bool, scale: float, row_chunk: int = 2048):
    """L = logsumexp of every score row (no V needed) [v1～v4 v2 §1]."""
    q, k = to_f64(q), to_f64(k)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    n = qh.shape[1]
    lse = np.empty(qh.shape[:2])
    for h in range(qh.shape[0]):
        for r0 in range(0, n, row_chunk):
            rows = np.arange(r0, min(n, r0 + row_chunk))
            s = _scores(qh[h], kh[h], rows, causal, float(scale))
            lse[h, rows] = _softmax_rows(s)[3]
    return lse.reshape(lead + lse.shape[1:])


def attention_abs_weighted_values(q, k, v, causal: bool, scale: float, rows=None,
                                  row_chunk: int = 2048):
    """A[i, c] = sum_j P_ij |V_jc|, with P = softmax(scale Q K^T) as in
    attention_forward [V1详解 §1.1]: the softmax average of |V| per row.

    Not a quantity of the method itself: it is the scale of the error that
    rounding the probabilities to a 16-bit format before the P V product
    adds to O (each P_ij carries a relative error of at most 2^-9 in bf16, so
    O_ic moves by at most 2^-9 (A_ic + |O_ic|) once normalised; the derivation
    is with the tolerances).  ``rows`` as in attention_forward_rows (None:
    every row).  Returns [..., R, d].
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    n = qh.shape[1]
    if rows is None:
        rows_all = np.arange(n)
        per_head = None
    else:
        rows_all = np.asarray(rows)
        per_head = rows_all.reshape(-1, rows_all.shape[-1]) if rows_all.ndim > 1 else None
    r = rows_all.shape[-1]
    out = np.empty((qh.shape[0], r, vh.shape[2]))
    for h in range(qh.shape[0]):
        rr = per_head[h] if per_head is not None else rows_all
        for r0 in range(0, r, row_chunk):
            sub = rr[r0:r0 + row_chunk]
            p = _softmax_rows(_scores(qh[h], kh[h], sub, causal, float(scale)))[0]
            out[h, r0:r0 + len(sub)] = p @ np.abs(vh[h])
    return out.reshape(lead + out.shape[1:])


# --------------------------------------------------------------------------
# attention backward: the gradient formulas
# --------------------------------------------------------------------------

def _head_backward_chunk(qh, kh, vh, doh, rows, causal, scale):
    """P, dP and dS for a set of full query rows of one head.

    [V1详解 §6.1]: dP = dO V^T and dS = P o (dP - rowsum(dP o P) 1^T).
    The row sum is taken from its definition, rowsum(dP o P); the identity
    rowsum(dP o P) = rowsum(dO o O) of the same section is checked
    separately by the tests, not assumed here.
    """
    s = _scores(qh, kh, rows, causal, scale)
    p = _softmax_rows(s)[0]
    dp = doh[rows] @ vh.T
    d_row = (dp * p).sum(axis=1)
    ds = p * (dp - d_row[:, None])
    return p, dp, ds, d_row


def attention_backward(q, k, v, do, causal: bool, scale: float):
    """Gradients of O = softmax(scale Q K^T) V w.r.t. Q, K, V given dO.

    Returns (dQ, dK, dV, D) with D the per-row sum rowsum(dP o P).

    [V1详解 §6.1] gives dV = P^T dO, dP = dO V^T and
    dS = P o (dP - rowsum(dP o P) 1^T).  The pages stop at dS; since
    S = scale Q K^T, the chain rule gives dQ = scale dS K and
    dK = scale dS^T Q (a reading recorded with the others).
    """
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    doh, _ = _heads(do)
    n = qh.shape[1]
    dq = np.empty_like(qh)
    dk = np.empty_like(kh)
    dv = np.empty_like(vh)
    dvec = np.empty(qh.shape[:2])
    rows = np.arange(n)
    for h in range(qh.shape[0]):
        p, _, ds, d_row = _head_backward_chunk(qh[h], kh[h], vh[h], doh[h], rows,
                                               causal, float(scale))
        dv[h] = p.T @ doh[h]
        dq[h] = float(scale) * (ds @ kh[h])
        dk[h] = float(scale) * (ds.T @ qh[h])
        dvec[h] = d_row
    shape = lambda a: a.reshape(lead + a.shape[1:])  # noqa: E731
    return shape(dq), shape(dk), shape(dv), shape(dvec)


def attention_backward_query_rows(q, k, v, do, rows, causal: bool, scale: float):
    """dQ for selected query rows only: dQ_R = scale dS_R K (each query row's
    gradient depends on that row's scores only).  ``rows`` as in
    attention_forward_rows.  Returns dQ [..., R, d]."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    doh, _ = _heads(do)
    rows = np.asarray(rows)
    per_head = rows.reshape(-1, rows.shape[-1]) if rows.ndim > 1 else None
    out = np.empty((qh.shape[0], rows.shape[-1], kh.shape[2]))
    for h in range(qh.shape[0]):
        rr = per_head[h] if per_head is not None else rows
        _, _, ds, _ = _head_backward_chunk(qh[h], kh[h], vh[h], doh[h], rr,
                                           causal, float(scale))
        out[h] = float(scale) * (ds @ kh[h])
    return out.reshape(lead + out.shape[1:])


def attention_backward_key_rows(q, k, v, do, key_rows, causal: bool, scale: float,
                                row_chunk: int = 1024):
    """dK and dV for selected key rows J only.

    dV_J = P[:, J]^T dO and dK_J = scale dS[:, J]^T Q need the columns J of
    P and dS over every query row, and each of those rows needs its full
    softmax; the query rows are walked in chunks of ``row_chunk`` and only
    the columns J are kept.  Returns (dK_J [..., R, d], dV_J [..., R, d]).
    """
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    doh, _ = _heads(do)
    key_rows = np.asarray(key_rows)
    per_head = key_rows.reshape(-1, key_rows.shape[-1]) if key_rows.ndim > 1 else None
    n = qh.shape[1]
    r = key_rows.shape[-1]
    dk = np.zeros((qh.shape[0], r, kh.shape[2]))
    dv = np.zeros((qh.shape[0], r, vh.shape[2]))
    for h in range(qh.shape[0]):
        jj = per_head[h] if per_head is not None else key_rows
        for r0 in range(0, n, row_chunk):
            rows = np.arange(r0, min(n, r0 + row_chunk))
            p, _, ds, _ = _head_backward_chunk(qh[h], kh[h], vh[h], doh[h], rows,
                                               causal, float(scale))
            dv[h] += p[:, jj].T @ doh[h][rows]
            dk[h] += float(scale) * (ds[:, jj].T @ qh[h][rows])
    return dk.reshape(lead + dk.shape[1:]), dv.reshape(lead + dv.shape[1:])


# --------------------------------------------------------------------------
# the tiled algorithms of the pages (fp64), used as pins of the definition
# --------------------------------------------------------------------------

def flash_forward_kv_outer_v1(q, k, v, block_r: int, block_c: int, causal: bool,
                              scale: float):
    """Tiled forward in the loop order and update form of [V1详解 §4.3, §5.1].

    Outer loop over K/V blocks j, inner loop over Q blocks i; the running
    O_i, m_i, l_i live in full-size arrays (the pages' HBM) between visits.
    Each step normalises immediately [V1详解 §5.1 step 5]:
        m_new = max(m_i, rowmax S_ij);  alpha = exp(m_i - m_new)
        l_new = alpha l_i + rowsum exp(S_ij - m_new)
        O_new = (alpha l_i / l_new) O_i + (1 / l_new) exp(S_ij - m_new) V_j
    Returns (O, m, l) with m, l the final row statistics.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    n, d = qh.shape[1], vh.shape[2]
    o = np.zeros((qh.shape[0], n, d))
    m = np.full((qh.shape[0], n), NEG_INF)
    l = np.zeros((qh.shape[0], n))
    for h in range(qh.shape[0]):
        for j0 in range(0, n, block_c):
            cols = np.arange(j0, min(n, j0 + block_c))
            kj, vj = kh[h][cols], vh[h][cols]
            for i0 in range(0, n, block_r):
                rows = np.arange(i0, min(n, i0 + block_r))
                s = float(scale) * (qh[h][rows] @ kj.T)
                if causal:
                    s = np.where(cols[None, :] <= rows[:, None], s, NEG_INF)
                m_i, l_i, o_i = m[h, rows], l[h, rows], o[h, rows]
                m_new = np.maximum(m_i, s.max(axis=1))
                live = np.isfinite(m_new)            # some key seen so far
                m_ref = np.where(live, m_new, 0.0)
                alpha = np.where(np.isfinite(m_i), np.exp(m_i - m_ref), 0.0)
                e = np.exp(s - m_ref[:, None])
                l_new = alpha * l_i + e.sum(axis=1)
                with np.errstate(divide="ignore", invalid="ignore"):
                    c_old = np.where(live, alpha * l_i / l_new, 0.0)
                    c_new = np.where(live, 1.0 / l_new, 0.0)
                o[h, rows] = c_old[:, None] * o_i + c_new[:, None] * (e @ vj)
                m[h, rows] = m_new
                l[h, rows] = l_new
    return (o.reshape(lead + o.shape[1:]), m.reshape(lead + m.shape[1:]),
            l.reshape(lead + l.shape[1:]))


def flash_forward_q_outer(q, k, v, block_r: int, block_c: int, causal: bool,
                          scale: float, tau_log2: float = 0.0):
    """Tiled forward, Q blocks outer, with deferred normalisation.

    Loop order of [A·FA §2.3] and [v1～v4 v1 §2 pseudocode]; the output is
    kept unnormalised and divided by l once at the end, and L = m + log l is
    returned instead of (m, l) [v1～v4 v2 §1]:
        m_new = max(m, rowmax S);  P~ = exp(S - m_new)
        l = exp(m - m_new) l + rowsum P~;  O = exp(m - m_new) O + P~ V_j
    With ``tau_log2`` > 0 the reference max is only moved when the row max
    rises by more than tau_log2 in log2 units, i.e. by a factor 2**tau_log2
    [v1～v4 v4 §3] (tau = log2 256 = 8 on the page); the result stays exact
    because the same reference is used for l and O.  Returns (O, L).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    qh, lead = _heads(q)
    kh, _ = _heads(k)
    vh, _ = _heads(v)
    n, d = qh.shape[1], vh.shape[2]
    thresh = float(tau_log2) * math.log(2.0)
    o_all = np.zeros((qh.shape[0], n, d))
    lse_all = np.zeros((qh.shape[0], n))
    for h in range(qh.shape[0]):
        for i0 in range(0, n, block_r):
            rows = np.arange(i0, min(n, i0 + block_r))
            qi = qh[h][rows]
            m = np.full(len(rows), NEG_INF)
            l = np.zeros(len(rows))
            o = np.zeros((len(rows), d))
            for j0 in range(0, n, block_c):
                cols = np.arange(j0, min(n, j0 + block_c))
                s = float(scale) * (qi @ kh[h][cols].T)
                if causal:
                    s = np.where(cols[None, :] <= rows[:, None], s, NEG_INF)
                row_max = s.max(axis=1)
                move = row_max > m + thresh if thresh > 0 else row_max > m
                move |= ~np.isfinite(m) & np.isfinite(row_max)
                m_new = np.where(move, row_max, m)
                # correction factor exp(m_old - m_new): 1 where the reference
                # stays, 0 where nothing had been accumulated yet
                alpha = np.ones(len(rows))
                moved_live = move & np.isfinite(m)
                alpha[moved_live] = np.exp(m[moved_live] - m_new[moved_live])
                alpha[move & ~np.isfinite(m)] = 0.0
                m_ref = np.where(np.isfinite(m_new), m_new, 0.0)
                p = np.exp(s - m_ref[:, None])
                l = alpha * l + p.sum(axis=1)
                o = alpha[:, None] * o + p @ vh[h][cols]
                m = m_new
            with np.errstate(divide="ignore", invalid="ignore"):
                o_all[h, rows] = np.where(l[:, None] > 0, o / l[:, None], 0.0)
                lse_all[h, rows] = np.where(l > 0, m + np.log(l), NEG_INF)
    return (o_all.reshape(lead + o_all.shape[1:]),
            lse_all.reshape(lead + lse_all.shape[1:]))
