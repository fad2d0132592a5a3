"""Backward parity: libfattn on the GPU vs the fp64 oracle's analytic
gradients on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import gather_rows, run_fwd, to_np
from tolerances import check_grad, check_l, check_o

pytestmark = pytest.mark.gpu


def run_fwd_bwd(inp, causal, scale):
    o, lse = run_fwd(inp, causal, scale)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
    status = A.fattn_check_status()
    assert status == 0, f"fattn status {status}"
    return dq, dk, dv


SMALL = [
    (1, 1, 128, 64, False),
    (1, 2, 200, 64, True),
    (2, 1, 1, 128, False),
    (1, 1, 1, 64, True),
    (1, 2, 129, 128, True),
    (1, 1, 257, 128, False),
    (2, 2, 333, 64, True),
    (1, 2, 640, 128, True),
    (1, 2, 1000, 128, False),
    (1, 1, 511, 64, False),
    # causal, even tile counts: every head dealt K/V tile by K/V tile
    # (small grids), and 64 paired heads followed by 16 single-tile heads
    (2, 4, 1024, 64, True),
    (4, 20, 512, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_bwd_small(B, H, N, d, causal):
    w = W.Workload("case", B, H, N, d, causal, seed=31 + N + d)
    inp = W.make_inputs(w)
    dq, dk, dv = run_fwd_bwd(inp, causal, w.scale)
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    check_grad(to_np(dq), gq, "dQ")
    check_grad(to_np(dk), gk, "dK")
    check_grad(to_np(dv), gv, "dV")


def test_bwd_outlier_rows_small():
    """Large-score rows (x20) as in the causal benchmark workload, at a size
    the oracle evaluates in full."""
    w = W.Workload("outl", 1, 2, 768, 128, True, outlier_frac=0.01, outlier_mult=20.0, seed=77)
    inp = W.make_inputs(w)
    dq, dk, dv = run_fwd_bwd(inp, True, w.scale)
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], True,
                                              w.scale)
    check_grad(to_np(dq), gq, "dQ")
    check_grad(to_np(dk), gk, "dK")
    check_grad(to_np(dv), gv, "dV")


def test_bwd_medium_d64_full():
    w = W.MEDIUM_D64
    inp = W.make_inputs(w)
    dq, dk, dv = run_fwd_bwd(inp, w.causal, w.scale)
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], w.causal,
                                              w.scale)
    check_grad(to_np(dq), gq, "dQ")
    check_grad(to_np(dk), gk, "dK")
    check_grad(to_np(dv), gv, "dV")


def _heads_subset(w, count, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(w.B * w.H, generator=g)[:count].tolist()


# Non-causal, 128 heads: the items run in several L2-sized head sections and
# every K/V tile starts its walk on a different Q tile.
SECTIONS_NONCAUSAL = W.Workload("b8h16_n2048_d128_sections", 8, 16, 2048, 128, False, seed=1006)
# The same with a ragged last tile (16 tiles, the last 80 rows long).
SECTIONS_RAGGED = W.Workload("b8h16_n2000_d128_sections", 8, 16, 2000, 128, False, seed=1008)
# Causal with an odd number of tiles: the items keep the all-heads order
# (no pairing); 64 heads, so several items of a head run at once.
CAUSAL_ODD_TILES = W.Workload("b4h16_n1920_d128_causal", 4, 16, 1920, 128, True, seed=1009)
# d = 64 with several head sections (256 heads).
SECTIONS_D64 = W.Workload("b8h32_n4096_d64_sections", 8, 32, 4096, 64, False, seed=1010)


@pytest.mark.parametrize("w,q_rows,k_rows,k_heads", [
    (SECTIONS_NONCAUSAL, 24, 16, 2),
    (SECTIONS_RAGGED, 24, 16, 2),
    (CAUSAL_ODD_TILES, 24, 16, 2),
    (SECTIONS_D64, 8, 16, 2),
])
def test_bwd_full_size_sampled(w, q_rows, k_rows, k_heads):
    """Full-size launches of the scheduling cases (head sections, ragged last
    tile, odd causal tile count, d = 64).  dQ is checked on seeded query rows
    of every head; dK, dV on seeded key rows of a few seeded heads (each
    needs the whole softmax of every query row of that head).  The per-tensor
    scale is the max |grad| over the checked rows.  The measured workloads
    are compared element by element in test_full_size_gpu.py."""
    inp = W.make_inputs(w)
    dq, dk, dv = run_fwd_bwd(inp, w.causal, w.scale)
    r = W.sample_rows(w, q_rows, seed=w.seed + 2)
    gq = oracle.attention_backward_query_rows(inp["q"], inp["k"], inp["v"], inp["do"],
                                              r.numpy(), w.causal, w.scale)
    check_grad(gather_rows(dq, r), gq, "dQ")
    heads = _heads_subset(w, k_heads, w.seed + 3)
    kr = W.sample_rows(w, k_rows, seed=w.seed + 4)
    for hflat in heads:
        b, h = divmod(hflat, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        sub = {n: inp[n][sl] for n in ("q", "k", "v", "do")}
        rows = kr[b, h].numpy()
        gk, gv = oracle.attention_backward_key_rows(sub["q"], sub["k"], sub["v"], sub["do"],
                                                    rows, w.causal, w.scale)
        check_grad(to_np(dk[sl])[0, 0, rows], gk[0, 0], f"dK head {hflat}")
        check_grad(to_np(dv[sl])[0, 0, rows], gv[0, 0], f"dV head {hflat}")
    # properties that hold at any size (P rows sum to one):
    # sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, per head
    dk64, dv64 = to_np(dk), to_np(dv)
    do64 = to_np(inp["do"])
    tol_k = 2.0 ** -7 * np.abs(dk64).sum(axis=2)
    tol_v = 2.0 ** -7 * np.abs(dv64).sum(axis=2) + 1e-6
    assert (np.abs(dk64.sum(axis=2)) <= tol_k).all()
    assert (np.abs(dv64.sum(axis=2) - do64.sum(axis=2)) <= tol_v).all()


def test_bwd_preprocess_entry_point():
    """fattn_bwd_preprocess: D = rowsum(dO o O) in fp32 and a zeroed dQ
    accumulator (random inputs, checked against an fp64 row sum)."""
    g = torch.Generator().manual_seed(5)
    o = torch.randn(2, 3, 77, 128, generator=g).to(torch.bfloat16)
    do = torch.randn(2, 3, 77, 128, generator=g).to(torch.bfloat16)
    D = torch.full((2, 3, 77), float("nan"), device="cuda")
    acc = torch.full((2, 3, 77, 128), float("nan"), device="cuda")
    A.fattn_bwd_preprocess(o.cuda(), do.cuda(), D, acc)
    assert A.fattn_check_status() == 0
    want = (to_np(o) * to_np(do)).sum(-1)
    assert np.abs(to_np(D) - want).max() <= 1e-4 * max(1.0, np.abs(want).max())
    assert bool((acc == 0).all())


def test_bwd_workspace_reuse_and_stream():
    """Two backward passes on a side stream with one caller-owned workspace
    give identical dK, dV (dQ sums atomically, so only its tolerance holds)."""
    w = W.Workload("ws", 1, 2, 300, 64, True, seed=8)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        o, lse = A.fattn_fwd(q, k, v, causal=True, scale=w.scale)
        ws = A.workspace_for(q)
        r1 = A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, workspace=ws)
        r1 = [t.clone() for t in r1]
        r2 = A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, workspace=ws)
    side.synchronize()
    assert A.fattn_check_status() == 0
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])
    gq, _, _, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], True, w.scale)
    check_grad(to_np(r2[0]), gq, "dQ")


def test_long_sequence_65536():
    """N = 65536 (512 tiles per head), causal: O, L and dQ on seeded rows of
    both heads against the oracle; dK, dV through the identities that hold at
    any size (the oracle's key rows would need every query row's softmax)."""
    w = W.Workload("b1h2_n65536_d128_causal", 1, 2, 65536, 128, True, seed=1007)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, True, w.scale)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
    assert A.fattn_check_status() == 0
    r = W.sample_rows(w, 24, seed=w.seed + 1)
    o_ref, l_ref = oracle.attention_forward_rows(inp["q"], inp["k"], inp["v"], r.numpy(), True,
                                                 w.scale)
    check_o(gather_rows(o, r), o_ref)
    check_l(gather_rows(lse, r), l_ref)
    gq = oracle.attention_backward_query_rows(inp["q"], inp["k"], inp["v"], inp["do"],
                                              r.numpy(), True, w.scale)
    check_grad(gather_rows(dq, r), gq, "dQ")
    dk64, dv64, do64 = to_np(dk), to_np(dv), to_np(inp["do"])
    assert (np.abs(dk64.sum(axis=2)) <= 2.0 ** -7 * np.abs(dk64).sum(axis=2)).all()
    assert (np.abs(dv64.sum(axis=2) - do64.sum(axis=2))
            <= 2.0 ** -7 * np.abs(dv64).sum(axis=2) + 1e-6).all()
