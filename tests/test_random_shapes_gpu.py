"""Forward and backward against the oracle on seeded random shapes: ragged
sequence lengths, both head dimensions, with and without the causal mask, so
that tile tails, single-tile and paired schedules and small grids mix in ways
the hand-picked cases do not."""

import random

import pytest

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import run_fwd, to_np
from tolerances import check_grad, check_l, check_o

pytestmark = pytest.mark.gpu


def _shapes(count, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(count):
        out.append((rng.randint(1, 2), rng.randint(1, 6), rng.randint(1, 1400),
                    rng.choice([64, 128]), rng.random() < 0.6))
    return out


@pytest.mark.parametrize("B,H,N,d,causal", _shapes(8, 424242))
def test_fwd_random_shape(B, H, N, d, causal):
    w = W.Workload("random", B, H, N, d, causal, backward=False, seed=5 * N + d)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, causal, w.scale)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], causal, w.scale)
    check_o(to_np(o), o_ref)
    check_l(to_np(lse), l_ref)


@pytest.mark.parametrize("B,H,N,d,causal", _shapes(8, 737373))
def test_bwd_random_shape(B, H, N, d, causal):
    w = W.Workload("random", B, H, N, d, causal, seed=7 * N + d)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=causal, scale=w.scale)
    dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    assert A.fattn_check_status() == 0
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    check_grad(to_np(dq), gq, "dQ")
    check_grad(to_np(dk), gk, "dK")
    check_grad(to_np(dv), gv, "dV")
