"""The CTA-pair backward kernel (d = 128, default mode) against the fp64
oracle and against the one-CTA-per-tile kernel on the same inputs: unit
boundaries (one tile, an odd tile count whose last unit has a rank-1 tile
past N, ragged N), causal and not, paired units with a balancing tail, and
several head sections."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import gather_rows, run_fwd, to_np
from tolerances import check_grad

pytestmark = pytest.mark.gpu


def _bwd(inp, causal, scale, o, lse, pair):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    A.fattn_set_bwd_pair(pair)
    try:
        out = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
        status = A.fattn_check_status()
    finally:
        A.fattn_set_bwd_pair(False)
    assert status == 0, f"status {status}"
    return out


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 1, 128, False),     # one tile: rank 1's tile lies wholly past N
    (1, 1, 1, True),
    (1, 2, 129, True),      # two tiles, the second holds one row
    (2, 3, 640, True),      # five tiles: the last unit's second tile is past N
    (1, 2, 1000, False),
    (1, 2, 333, True),
    (4, 20, 512, True),     # paired units plus single units at the end
    (2, 4, 1536, False),
])
def test_pair_backward_matches_oracle_and_single_cta(B, H, N, causal):
    w = W.Workload("pair", B, H, N, 128, causal, seed=4100 + N + B)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, causal, w.scale)
    pair = _bwd(inp, causal, w.scale, o, lse, True)
    single = _bwd(inp, causal, w.scale, o, lse, False)
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    for got, ref, name in zip(pair, (gq, gk, gv), ("dQ", "dK", "dV")):
        check_grad(to_np(got), ref, f"{name} (pair)")
    for a, b, name in zip(pair, single, ("dQ", "dK", "dV")):
        a64, b64 = to_np(a), to_np(b)
        rel = np.abs(a64 - b64).max() / max(np.abs(b64).max(), 1e-4)
        assert rel <= 2.0 ** -6, f"{name}: pair vs single-CTA kernel differ by {rel:.3e}"


def test_pair_backward_full_size_sections():
    """Non-causal, 128 heads in several L2 head sections (full-size launch):
    dQ on seeded query rows of every head, dK and dV of two seeded heads in
    full, against the oracle."""
    w = W.Workload("pair_sections", 8, 16, 2048, 128, False, seed=4300)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, False, w.scale)
    dq, dk, dv = _bwd(inp, False, w.scale, o, lse, True)
    r = W.sample_rows(w, 16, seed=w.seed + 1)
    gq = oracle.attention_backward_query_rows(inp["q"], inp["k"], inp["v"], inp["do"],
                                              r.numpy(), False, w.scale)
    check_grad(gather_rows(dq, r), gq, "dQ rows (pair)")
    for hflat in (5, 100):
        b, h = divmod(hflat, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        sub = {n: inp[n][sl] for n in ("q", "k", "v", "do")}
        _, gk, gv, _ = oracle.attention_backward(sub["q"], sub["k"], sub["v"], sub["do"], False,
                                                 w.scale)
        check_grad(to_np(dk[sl]), gk, f"dK head {hflat} (pair)")
        check_grad(to_np(dv[sl]), gv, f"dV head {hflat} (pair)")
