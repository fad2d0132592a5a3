"""Checks that pin the fp64 oracle to facts fixed outside itself.

Each check takes the oracle module (so that the mutation tests can hand in a
deliberately broken copy) and raises AssertionError when the oracle disagrees
with the fact.  The facts come from the source pages (a printed worked
example, stated invariants and identities), from closed forms of special
inputs, from central finite differences, and from an independent library
routine (torch's CPU scaled_dot_product_attention in fp64).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, shape, scale_in=1.0):
    r = _rng(seed)
    return tuple(scale_in * r.standard_normal(shape) for _ in range(4))


# ---------------------------------------------------------------- page values

def check_worked_example(o):
    """FlashAttention v1～v4, v1 §2: blocks [1,2] then [0,3] give m1=2,
    l1=e^-1+1, then m2=3, l2=e^-2+e^-1+e^-3+1."""
    with open(os.path.join(GOLDEN, "worked_example_online_softmax.json")) as f:
        g = json.load(f)
    x = [v for b in g["blocks"] for v in b]
    _, m, l, hist = o.online_softmax_blockwise(x, len(g["blocks"][0]))
    env = {"exp": math.exp}
    for (hm, hl), want in zip(hist, g["after_each_block"]):
        assert hm == want["m"]
        assert abs(hl - eval(want["l"], env)) <= 1e-15 * abs(hl)
        assert abs(hl - eval(want["l_simplified"], env)) <= 1e-15 * abs(hl)
    # the page's claim: the final l is the sum over the whole vector minus 3
    assert abs(l - sum(math.exp(v - 3) for v in x)) <= 1e-15 * l
    # the same numbers as an attention instance: q = 1, keys 1,2,0,3, d = 1;
    # V = identity makes O equal to the softmax row itself
    q = np.ones((1, 1))
    k = np.array(x, dtype=np.float64)[:, None]
    v = np.eye(4)
    out, lse = o.attention_forward(q, k, v, False, 1.0)
    l2 = eval(g["after_each_block"][1]["l_simplified"], env)
    assert abs(lse[0] - (3.0 + math.log(l2))) <= 1e-14
    want = np.array([math.exp(t - 3.0) / l2 for t in x])
    assert np.abs(out[0] - want).max() <= 1e-15


# ---------------------------------------------------------------- softmax

def check_three_pass_vs_library(o):
    """Three-pass safe softmax [V1详解 §3.1] equals scipy's softmax."""
    from scipy.special import logsumexp, softmax

    r = _rng(1)
    for n in (1, 2, 7, 64):
        x = 3.0 * r.standard_normal(n)
        y, m, l = o.softmax_three_pass(x)
        assert np.abs(y - softmax(x)).max() <= 1e-15
        assert abs(m + math.log(l) - logsumexp(x)) <= 1e-13
        assert abs(y.sum() - 1.0) <= 1e-14


def check_blockwise_equals_three_pass(o):
    """Online softmax at every block size equals three-pass softmax
    [V1详解 §3.3]: the rescaling identity is exact, so only rounding differs."""
    r = _rng(2)
    for n in (1, 5, 17):
        x = 4.0 * r.standard_normal(n)
        y3, m3, l3 = o.softmax_three_pass(x)
        for b in range(1, n + 1):
            y, m, l, _ = o.online_softmax_blockwise(x, b)
            assert m == m3
            assert abs(l - l3) <= 1e-12 * l3
            assert np.abs(y - y3).max() <= 1e-12


# ---------------------------------------------------------------- closed forms

def check_closed_forms(o):
    """Special inputs with a known answer.

    * N = 1: O = V and L = scale q.k (softmax of a single score is 1).
    * identical key rows: every visible key has the same score, P is uniform,
      O_i = mean of the visible V rows, L_i = scale q_i.k + log(#visible).
    * causal row 0 sees only key 0: O_0 = V_0, L_0 = scale q_0.k_0.
    """
    r = _rng(3)
    q, k, v = (r.standard_normal((2, 1, 1, 5)) for _ in range(3))
    out, lse = o.attention_forward(q, k, v, False, 0.7)
    assert np.abs(out - v).max() <= 1e-15
    assert np.abs(lse - 0.7 * (q * k).sum(-1)).max() <= 1e-14

    n, d = 9, 4
    q = r.standard_normal((1, 2, n, d))
    krow = r.standard_normal(d)
    k = np.broadcast_to(krow, (1, 2, n, d)).copy()
    v = r.standard_normal((1, 2, n, d))
    for causal in (False, True):
        out, lse = o.attention_forward(q, k, v, causal, 0.5)
        for i in range(n):
            vis = i + 1 if causal else n
            assert np.abs(out[..., i, :] - v[..., :vis, :].mean(-2)).max() <= 1e-14
            want = 0.5 * (q[..., i, :] @ krow) + math.log(vis)
            assert np.abs(lse[..., i] - want).max() <= 1e-13

    q, k, v = (r.standard_normal((1, 3, 6, 4)) for _ in range(3))
    out, lse = o.attention_forward(q, k, v, True, 0.9)
    assert np.abs(out[..., 0, :] - v[..., 0, :]).max() <= 1e-15
    assert np.abs(lse[..., 0] - 0.9 * (q[..., 0, :] * k[..., 0, :]).sum(-1)).max() <= 1e-14


def check_one_hot_closed_form(o):
    """K = identity (d = N) and q_i = c e_pi(i): the scores are c on the
    key pi(i) and 0 elsewhere, so
        O_i = (e^c V_pi(i) + sum_{j != pi(i)} V_j) / (e^c + N - 1),
        L_i = log(e^c + N - 1).
    Fixes which operand is transposed and which rows of V are mixed."""
    n = 6
    r = _rng(4)
    perm = r.permutation(n)
    c = 2.5
    q = c * np.eye(n)[perm][None, None]
    k = np.eye(n)[None, None]
    v = r.standard_normal((1, 1, n, 3))
    out, lse = o.attention_forward(q, k, v, False, 1.0)
    for i in range(n):
        j = perm[i]
        want = (math.exp(c) * v[0, 0, j] + v[0, 0].sum(0) - v[0, 0, j]) / (math.exp(c) + n - 1)
        assert np.abs(out[0, 0, i] - want).max() <= 1e-14
        assert abs(lse[0, 0, i] - math.log(math.exp(c) + n - 1)) <= 1e-14


def check_large_scores_stable(o):
    """Scores of size 1e4 neither overflow nor lose the answer [V1详解 §5.3]:
    with the one-hot construction at c = 1e4 the weight of the matching key
    is 1 to within exp(-1e4), so O_i = V_pi(i) and L_i = c."""
    n = 5
    r = _rng(5)
    perm = r.permutation(n)
    c = 1.0e4
    q = c * np.eye(n)[perm][None, None]
    k = np.eye(n)[None, None]
    v = r.standard_normal((1, 1, n, 2))
    for sign in (1.0, -1.0):
        out, lse = o.attention_forward(sign * q, k, v, False, 1.0)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        if sign > 0:
            assert np.abs(out[0, 0] - v[0, 0, perm]).max() <= 1e-12
            assert np.abs(lse[0, 0] - c).max() <= 1e-9
        else:
            # score -c on the matching key, 0 on the rest: mean of the others
            for i in range(n):
                others = np.delete(v[0, 0], perm[i], axis=0)
                assert np.abs(out[0, 0, i] - others.mean(0)).max() <= 1e-12


# ---------------------------------------------------------------- invariants

def check_invariants(o):
    """Invariances that the pages' softmax implies.

    * rows of P sum to 1 [v1～v4 v1 §2]: with V = all ones, O = all ones.
    * shift invariance [A·FA §4]: K <- K + 1 u^T adds scale q_i.u to every
      score of row i, so O is unchanged and L_i grows by scale q_i.u
      (masked or not).
    * non-causal: permuting the rows of K and V together changes nothing;
      permuting the rows of Q permutes the rows of O and L.
    """
    r = _rng(6)
    q, k, v = (r.standard_normal((2, 2, 11, 4)) for _ in range(3))
    sc = 0.45
    for causal in (False, True):
        out1, _ = o.attention_forward(q, k, np.ones_like(v), causal, sc)
        assert np.abs(out1 - 1.0).max() <= 1e-14
        out, lse = o.attention_forward(q, k, v, causal, sc)
        u = r.standard_normal(4)
        out_s, lse_s = o.attention_forward(q, k + u, v, causal, sc)
        assert np.abs(out_s - out).max() <= 1e-13
        assert np.abs(lse_s - (lse + sc * (q @ u))).max() <= 1e-12
    out, lse = o.attention_forward(q, k, v, False, sc)
    p = r.permutation(11)
    out_p, lse_p = o.attention_forward(q, k[..., p, :], v[..., p, :], False, sc)
    assert np.abs(out_p - out).max() <= 1e-13
    assert np.abs(lse_p - lse).max() <= 1e-13
    out_q, lse_q = o.attention_forward(q[..., p, :], k, v, False, sc)
    assert np.abs(out_q - out[..., p, :]).max() <= 1e-13
    assert np.abs(lse_q - lse[..., p]).max() <= 1e-13


def check_causal_prefix(o):
    """Causal row i is ordinary attention of query i over keys 0..i."""
    r = _rng(7)
    q, k, v = (r.standard_normal((1, 1, 8, 3)) for _ in range(3))
    out, lse = o.attention_forward(q, k, v, True, 0.8)
    for i in range(8):
        oi, li = o.attention_forward(q[..., i:i + 1, :], k[..., :i + 1, :],
                                     v[..., :i + 1, :], False, 0.8)
        assert np.abs(out[..., i, :] - oi[..., 0, :]).max() <= 1e-14
        assert np.abs(lse[..., i] - li[..., 0]).max() <= 1e-14


# ---------------------------------------------------------------- library

def check_against_torch_sdpa(o):
    """torch's CPU scaled_dot_product_attention in fp64 (and its autograd
    gradients) is an independent implementation of the same definition."""
    import torch

    r = _rng(8)
    shape = (2, 3, 13, 5)
    q, k, v, do = (r.standard_normal(shape) for _ in range(4))
    for causal in (False, True):
        t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
        out_t = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal,
                                                                 scale=0.37)
        out_t.backward(torch.tensor(do))
        out, _ = o.attention_forward(q, k, v, causal, 0.37)
        dq, dk, dv, _ = o.attention_backward(q, k, v, do, causal, 0.37)
        assert np.abs(out - out_t.detach().numpy()).max() <= 1e-13
        for mine, ref in ((dq, t[0].grad), (dk, t[1].grad), (dv, t[2].grad)):
            assert np.abs(mine - ref.numpy()).max() <= 1e-12
        # L against logsumexp of the library's own score matrix
        s = 0.37 * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(13, 13, dtype=torch.bool).triu(1), float("-inf"))
        _, lse = o.attention_forward(q, k, v, causal, 0.37)
        assert np.abs(lse - torch.logsumexp(s, -1).numpy()).max() <= 1e-13


# ---------------------------------------------------------------- gradients

def check_finite_differences(o):
    """Central finite differences of f = sum(O o dO) with respect to every
    entry of Q, K and V agree with the analytic gradients."""
    r = _rng(9)
    for causal in (False, True):
        for n, d in ((3, 2), (6, 4)):
            q, k, v, do = (r.standard_normal((1, 1, n, d)) for _ in range(4))
            sc = 0.6
            dq, dk, dv, _ = o.attention_backward(q, k, v, do, causal, sc)

            def f(qq, kk, vv):
                return float((o.attention_forward(qq, kk, vv, causal, sc)[0] * do).sum())

            h = 1e-5
            for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
                num = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += h
                    xm[idx] -= h
                    args_p = {"q": q, "k": k, "v": v}
                    args_m = dict(args_p)
                    args_p[name], args_m[name] = xp, xm
                    num[idx] = (f(args_p["q"], args_p["k"], args_p["v"])
                                - f(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
                err = np.abs(num - g).max() / max(1e-12, np.abs(g).max())
                assert err <= 1e-7, (name, causal, n, d, err)


def check_backward_identities(o):
    """[V1详解 §6.1]: rowsum(dP o P) = rowsum(dO o O) (the D identity).
    Because every row of P sums to 1, every row of dS sums to 0, so
    sum_j dK_j = 0; and sum_j dV_j = sum_j (P^T dO)_j = sum_i dO_i."""
    r = _rng(10)
    q, k, v, do = (r.standard_normal((2, 2, 12, 4)) for _ in range(4))
    for causal in (False, True):
        out, _ = o.attention_forward(q, k, v, causal, 0.5)
        dq, dk, dv, dvec = o.attention_backward(q, k, v, do, causal, 0.5)
        assert np.abs(dvec - (do * out).sum(-1)).max() <= 1e-13
        assert np.abs(dk.sum(-2)).max() <= 1e-13
        assert np.abs(dv.sum(-2) - do.sum(-2)).max() <= 1e-13


# ---------------------------------------------------------------- algorithms

def check_tiled_algorithms(o):
    """The pages' tiled algorithms give the definition's result at every
    tiling: K/V-outer with per-step normalisation [V1详解 §5.2], Q-outer with
    deferred normalisation [v1～v4 v2 §1], and conditional rescaling with
    tau = 8 [v1～v4 v4 §3]."""
    r = _rng(11)
    n = 13
    q, k, v = (r.standard_normal((1, 2, n, 3)) for _ in range(3))
    q[..., 4, :] *= 20.0                       # a row with large scores
    for causal in (False, True):
        out, lse = o.attention_forward(q, k, v, causal, 0.7)
        for br, bc in ((1, 1), (2, 3), (4, 5), (13, 13), (5, 13), (13, 2)):
            o1, m1, l1 = o.flash_forward_kv_outer_v1(q, k, v, br, bc, causal, 0.7)
            assert np.abs(o1 - out).max() <= 1e-12
            assert np.abs(m1 + np.log(l1) - lse).max() <= 1e-12
            for tau in (0.0, 8.0):
                o2, l2 = o.flash_forward_q_outer(q, k, v, br, bc, causal, 0.7, tau)
                assert np.abs(o2 - out).max() <= 1e-12
                assert np.abs(l2 - lse).max() <= 1e-12


def check_row_subsets(o):
    """The row-subset entry points (used at long sequence lengths) return
    the same rows as the full computation (checked against the full one
    after the full one is pinned by the checks above)."""
    r = _rng(12)
    q, k, v, do = (r.standard_normal((1, 2, 19, 4)) for _ in range(4))
    rows = np.array([[0, 7, 18], [3, 4, 11]])
    for causal in (False, True):
        out, lse = o.attention_forward(q, k, v, causal, 0.5)
        dq, dk, dv, _ = o.attention_backward(q, k, v, do, causal, 0.5)
        orr, lrr = o.attention_forward_rows(q, k, v, rows[None], causal, 0.5)
        lall = o.attention_lse_all_rows(q, k, causal, 0.5, row_chunk=5)
        dqr = o.attention_backward_query_rows(q, k, v, do, rows[None], causal, 0.5)
        dkr, dvr = o.attention_backward_key_rows(q, k, v, do, rows[None], causal, 0.5,
                                                 row_chunk=4)
        for h in range(2):
            assert np.abs(orr[0, h] - out[0, h, rows[h]]).max() <= 1e-14
            assert np.abs(lrr[0, h] - lse[0, h, rows[h]]).max() <= 1e-14
            assert np.abs(dqr[0, h] - dq[0, h, rows[h]]).max() <= 1e-14
            assert np.abs(dkr[0, h] - dk[0, h, rows[h]]).max() <= 1e-13
            assert np.abs(dvr[0, h] - dv[0, h, rows[h]]).max() <= 1e-13
        assert np.abs(lall - lse).max() <= 1e-14


def check_abs_weighted_values(o):
    """sum_j P_ij |V_jc| (the scale of the P-rounding term in the O
    tolerance): with every V entry >= 0 it is O itself; with one key's value
    row e_c and the others zero it is that key's softmax weight (causal row
    0: exactly 1); with V of one sign flipped it does not change; and it
    bounds |O| from above.  Rows variant = full computation."""
    r = _rng(13)
    q, k = (r.standard_normal((1, 2, 17, 4)) for _ in range(2))
    v = r.standard_normal((1, 2, 17, 4))
    for causal in (False, True):
        a = o.attention_abs_weighted_values(q, k, v, causal, 0.6, row_chunk=5)
        out, _ = o.attention_forward(q, k, np.abs(v), causal, 0.6)
        assert np.abs(a - out).max() <= 1e-14
        assert np.abs(o.attention_abs_weighted_values(q, k, -v, causal, 0.6) - a).max() <= 1e-14
        signed, _ = o.attention_forward(q, k, v, causal, 0.6)
        assert (np.abs(signed) <= a + 1e-14).all()
        onehot = np.zeros_like(v)
        onehot[:, :, 0, 2] = -3.0
        a1 = o.attention_abs_weighted_values(q, k, onehot, causal, 0.6)
        s = 0.6 * np.einsum("bhid,bhjd->bhij", q, k)
        if causal:
            s = np.where(np.tril(np.ones((17, 17), bool)), s, -np.inf)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        assert np.abs(a1[..., 2] - 3.0 * p[..., 0]).max() <= 1e-14
        assert np.abs(a1[..., [0, 1, 3]]).max() == 0.0
        if causal:
            assert a1[0, 0, 0, 2] == 3.0
        rows = np.array([[0, 5, 16], [2, 3, 9]])
        ar = o.attention_abs_weighted_values(q, k, v, causal, 0.6, rows=rows[None])
        for h in range(2):
            assert np.abs(ar[0, h] - a[0, h, rows[h]]).max() <= 1e-14


ALL_CHECKS = [
    check_worked_example,
    check_three_pass_vs_library,
    check_blockwise_equals_three_pass,
    check_closed_forms,
    check_one_hot_closed_form,
    check_large_scores_stable,
    check_invariants,
    check_causal_prefix,
    check_against_torch_sdpa,
    check_finite_differences,
    check_backward_identities,
    check_tiled_algorithms,
    check_row_subsets,
    check_abs_weighted_values,
]
