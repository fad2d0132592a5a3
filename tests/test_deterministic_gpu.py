"""Deterministic backward ("FlashAttention v1～v4" v4 §4: cross-CTA dQ
reductions in a fixed order through semaphores): the gradients still match
the fp64 oracle, and repeated runs agree bit for bit."""

import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import run_fwd, to_np
from tolerances import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture
def deterministic():
    A.fattn_set_deterministic(True)
    try:
        yield
    finally:
        A.fattn_set_deterministic(False)


def _bwd(inp, causal, scale, o, lse, ws):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    out = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=scale, workspace=ws)
    assert A.fattn_check_status() == 0
    return out


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 4, 1024, 128, True),     # every K/V tile of a head in flight at once
    (2, 3, 777, 64, False),      # ragged tail, d = 64
    (1, 2, 1000, 128, False),
])
def test_deterministic_matches_oracle_and_repeats(deterministic, B, H, N, d, causal):
    w = W.Workload("det", B, H, N, d, causal, seed=500 + N + d)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, causal, w.scale)
    ws = A.workspace_for(o)
    runs = [_bwd(inp, causal, w.scale, o, lse, ws) for _ in range(3)]
    for other in runs[1:]:
        for a, b, name in zip(runs[0], other, ("dQ", "dK", "dV")):
            assert torch.equal(a, b), f"{name} differs between deterministic runs"
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    dq, dk, dv = runs[0]
    check_grad(to_np(dq), gq, "dQ")
    check_grad(to_np(dk), gk, "dK")
    check_grad(to_np(dv), gv, "dV")


def test_deterministic_many_items_per_cta():
    """Several work items per CTA (1024 items over at most 152 CTAs), causal:
    repeated deterministic runs agree bit for bit, and agree with the default
    (arrival-order) accumulation to fp32 rounding."""
    w = W.Workload("det_big", 2, 32, 2048, 128, True, seed=611)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, True, w.scale)
    ws = A.workspace_for(o)
    free = _bwd(inp, True, w.scale, o, lse, ws)
    A.fattn_set_deterministic(True)
    try:
        a = _bwd(inp, True, w.scale, o, lse, ws)
        b = _bwd(inp, True, w.scale, o, lse, ws)
    finally:
        A.fattn_set_deterministic(False)
    for x, y, name in zip(a, b, ("dQ", "dK", "dV")):
        assert torch.equal(x, y), f"{name} differs between deterministic runs"
    assert torch.equal(a[1], free[1]) and torch.equal(a[2], free[2])   # dK, dV never depend on it
    dq_a, dq_f = a[0].float(), free[0].float()
    rel = ((dq_a - dq_f).abs().max() / dq_f.abs().max()).item()
    assert rel < 1e-2, rel


def test_deterministic_repeats_on_the_benchmark_shape():
    """Forty deterministic backward passes on the causal N = 4096 workload
    (2048 items over the persistent grid): every one completes without a
    wait timeout and all agree bit for bit."""
    w = W.CAUSAL_OUTLIERS
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, True, w.scale)
    ws = A.workspace_for(o)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    A.fattn_set_deterministic(True)
    try:
        ref = None
        for it in range(40):
            A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, workspace=ws,
                        dq=dq, dk=dk, dv=dv)
            status = A.fattn_check_status()
            assert status == 0, f"run {it}: status {status}"
            if ref is None:
                ref = (dq.clone(), dk.clone(), dv.clone())
            else:
                for a, b, name in zip((dq, dk, dv), ref, ("dQ", "dK", "dV")):
                    assert torch.equal(a, b), f"run {it}: {name} differs"
    finally:
        A.fattn_set_deterministic(False)


def test_deterministic_with_concurrent_work_on_the_gpu():
    """The ordered backward waits on dQ adds of other CTAs of its grid, so all
    of them must be resident at once.  It is launched cooperatively: while a
    side stream keeps the SMs busy with matrix products, the result is either
    bit-identical to an uncontended run or a clean launch error, never a wait
    timeout.  The wait budget is cut to ~1/60 s for the test, so a grid that
    started only partly would time out well within it."""
    w = W.Workload("det_busy", 2, 32, 2048, 128, True, seed=612)
    inp = W.make_inputs(w)
    o, lse = run_fwd(inp, True, w.scale)
    ws = A.workspace_for(o)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    A.fattn_set_deterministic(True)
    A.fattn_set_wait_budget(1 << 25)
    try:
        ref = _bwd(inp, True, w.scale, o, lse, ws)
        ref = tuple(t.clone() for t in ref)
        for trial in range(3):
            torch.cuda.synchronize()
            with torch.cuda.stream(side):
                for _ in range(60):
                    a = (a @ a).mul_(1e-4)
            try:
                got = A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, workspace=ws)
            except RuntimeError as exc:          # refused up front: acceptable
                assert "CUDA error" in str(exc), str(exc)
                torch.cuda.synchronize()
                continue
            status = A.fattn_check_status()
            torch.cuda.synchronize()
            assert status == 0, f"trial {trial}: status {status}"
            for x, y, name in zip(got, ref, ("dQ", "dK", "dV")):
                assert torch.equal(x, y), f"trial {trial}: {name} differs"
    finally:
        A.fattn_set_wait_budget(0)
        A.fattn_set_deterministic(False)
        torch.cuda.synchronize()
