"""Forward parity: libfattn on the GPU vs the fp64 oracle on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import gather_rows, run_fwd, to_np
from tolerances import check_l, check_o

pytestmark = pytest.mark.gpu

# (B, H, N, d, causal): single tile, ragged tails, a lone row, several tile
# pairs, d = 64 and 128.
SMALL = [
    (1, 1, 128, 64, False),
    (1, 2, 200, 64, True),
    (2, 1, 1, 128, False),
    (1, 1, 1, 64, True),
    (1, 2, 129, 128, True),
    (1, 1, 257, 128, False),
    (2, 2, 333, 64, True),
    (1, 3, 640, 128, True),
    (1, 1, 64, 128, False),
    (1, 2, 1000, 128, False),
    (1, 1, 511, 64, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_fwd_small(B, H, N, d, causal):
    w = W.Workload("case", B, H, N, d, causal, backward=False, seed=17 + N + d)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, causal, w.scale)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], causal, w.scale)
    check_o(to_np(o), o_ref)
    check_l(to_np(lse), l_ref)


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_rescale_threshold_exact(tau, d):
    """Conditional rescaling ("FlashAttention v1～v4" v4 §3) is exact at any
    threshold: large-score rows force many max changes."""
    w = W.Workload("resc", 1, 2, 700, d, True, outlier_frac=0.05, outlier_mult=20.0,
                   backward=False, seed=99)
    inp = W.make_inputs(w)
    A.fattn_set_rescale_threshold(tau)
    try:
        o, lse = run_fwd(inp, True, w.scale)
    finally:
        A.fattn_set_rescale_threshold(-1.0)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], True, w.scale)
    check_o(to_np(o), o_ref)
    check_l(to_np(lse), l_ref)


def test_fwd_tiny_workload():
    w = W.TINY
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, w.causal, w.scale)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], w.causal, w.scale)
    check_o(to_np(o), o_ref)
    check_l(to_np(lse), l_ref)


def test_fwd_medium_d64_full():
    w = W.MEDIUM_D64
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, w.causal, w.scale)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], w.causal, w.scale)
    check_o(to_np(o), o_ref)
    check_l(to_np(lse), l_ref)


@pytest.mark.parametrize("w,rows", [(W.Workload("b8h32_n4096_d64_sections", 8, 32, 4096, 64,
                                                False, backward=False, seed=1010), 8)])
def test_fwd_full_size_sampled_rows(w, rows):
    """Full-size launch with 256 heads in several L2 head sections; the oracle
    evaluates a seeded sample of rows per head (always including the first
    and the last row).  The measured workloads are compared element by
    element in test_full_size_gpu.py."""
    inp = W.make_inputs(w, with_grad=False)
    o, lse = run_fwd(inp, w.causal, w.scale)
    r = W.sample_rows(w, rows, seed=w.seed + 1)
    o_ref, l_ref = oracle.attention_forward_rows(inp["q"], inp["k"], inp["v"], r.numpy(),
                                                 w.causal, w.scale)
    check_o(gather_rows(o, r), o_ref)
    check_l(gather_rows(lse, r), l_ref)
    assert np.isfinite(to_np(lse)).all()


def test_fwd_deterministic():
    w = W.Workload("det", 1, 4, 1024, 128, True, backward=False, seed=5)
    inp = W.make_inputs(w)
    o1, l1 = run_fwd(inp, True, w.scale)
    o2, l2 = run_fwd(inp, True, w.scale)
    assert torch.equal(o1, o2)
    assert (l1 == l2).all()


def test_fwd_key_value_permutation_invariance():
    """Non-causal attention does not depend on the order of the keys: permuting
    the rows of K and V together leaves O and L unchanged up to rounding
    order (checked on GPU outputs against each other, at any size)."""
    w = W.Workload("perm", 2, 2, 900, 128, False, backward=False, seed=3)
    inp = W.make_inputs(w)
    perm = torch.randperm(900, generator=torch.Generator().manual_seed(4))
    shuffled = dict(inp)
    shuffled["k"] = inp["k"][:, :, perm].contiguous()
    shuffled["v"] = inp["v"][:, :, perm].contiguous()
    o1, l1 = run_fwd(inp, False, w.scale)
    o2, l2 = run_fwd(shuffled, False, w.scale)
    assert np.abs(to_np(l2) - to_np(l1)).max() <= 1e-4
    assert np.abs(to_np(o2) - to_np(o1)).max() <= 1e-2


def test_status_ok_after_launches():
    assert A.fattn_check_status() == 0
