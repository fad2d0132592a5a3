"""fattn_bwd_noalloc, the backward pass for callers that cannot allocate
device memory at the point of the call (a plugin whose host framework owns
every allocation, a loop that cannot afford cudaMalloc's implicit
synchronisation, a caller without a spare buffer).  Its scratch is a fixed
array inside the library, so the call itself allocates nothing.

It must give the oracle's gradients, and what fattn_bwd gives with a
caller-owned workspace, on every call: the array keeps the previous call's
contents, and a second call in a row must not be affected by them.  This
file is collected last on purpose.
"""

import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import _lib
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import to_np
from tolerances import check_grad

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, scale):
    B, H, N, d = q.shape
    return lib.fattn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, N, d, int(causal), scale,
                                 torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 333, 64, True), (2, 4, 1024, 128, False)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(B, H, N, d, causal):
    """Two calls in a row, each against the fp64 oracle and against fattn_bwd
    with a caller-owned workspace.  dK and dV involve no cross-CTA sums, so
    they must be bit-identical to fattn_bwd's; dQ is summed by reduce-adds
    in arrival order, so it may differ from fattn_bwd's by fp32 reordering
    only (a stale accumulator would add a whole extra gradient)."""
    lib = _lib.load()
    w = W.Workload("noalloc", B, H, N, d, causal, seed=2024 + N)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=causal, scale=w.scale)
    ref_dq, ref_dk, ref_dv = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    assert A.fattn_check_status() == 0
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, w.scale)
        assert rc == _lib.FATTN_OK, _lib.status_string(rc)
        assert A.fattn_check_status() == 0
        check_grad(to_np(dq), gq, "dQ (no-alloc)")
        check_grad(to_np(dk), gk, "dK (no-alloc)")
        check_grad(to_np(dv), gv, "dV (no-alloc)")
        assert torch.equal(dk, ref_dk) and torch.equal(dv, ref_dv)
        rel = ((dq.float() - ref_dq.float()).abs().max() / ref_dq.float().abs().max()).item()
        assert rel <= 2.0 ** -7, rel


def test_noalloc_deterministic_twice():
    """Deterministic mode keeps its ordering counters in the built-in scratch
    too; every call must start them from zero, so two calls in a row give
    bit-identical dQ, dK, dV, equal to fattn_bwd's deterministic result."""
    lib = _lib.load()
    w = W.Workload("noalloc_det", 1, 4, 1024, 128, True, seed=2077)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=True, scale=w.scale)
    A.fattn_set_deterministic(True)
    try:
        ref = A.fattn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
        assert A.fattn_check_status() == 0
        for _ in range(2):
            got = tuple(torch.full_like(q, float("nan")) for _ in range(3))
            rc = _noalloc(lib, q, k, v, o, do, lse, *got, True, w.scale)
            assert rc == _lib.FATTN_OK, _lib.status_string(rc)
            assert A.fattn_check_status() == 0
            for a, b, name in zip(got, ref, ("dQ", "dK", "dV")):
                assert torch.equal(a, b), f"{name} differs from the deterministic fattn_bwd"
    finally:
        A.fattn_set_deterministic(False)
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], True,
                                              w.scale)
    check_grad(to_np(got[0]), gq, "dQ (no-alloc, ordered)")
    check_grad(to_np(got[1]), gk, "dK (no-alloc, ordered)")
    check_grad(to_np(got[2]), gv, "dV (no-alloc, ordered)")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, N, d = 1, 64, 4096, 128          # needs ~136 MB of scratch
    assert lib.fattn_bwd_workspace_bytes(B, H, N, d) > _lib.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = t.data_ptr()
    rc = lib.fattn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0, 0.088,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.FATTN_ERR_TOO_LARGE
    assert A.fattn_check_status() == 0
