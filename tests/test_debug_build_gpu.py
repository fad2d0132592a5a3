"""Small-shape parity on the checked debug variant of the library: every
kernel range-checks its computed indices (a failed check would report
FATTN_ERR_DEBUG_CHECK), and the forward's K/V ring runs with two stages, so
that its phases wrap every key tile pair.  The results must still match the
oracle, and no check may fire."""

import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import _lib, build
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import to_np
from tolerances import check_grad, check_l, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    lib = _lib.load(build.build(debug=True))
    saved = _lib._lib
    _lib._lib = lib
    try:
        yield lib
    finally:
        _lib._lib = saved


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 200, 64, True),
    (1, 2, 129, 128, True),
    (2, 1, 333, 128, False),
    (1, 3, 640, 64, False),
    (1, 2, 1000, 128, True),
])
@pytest.mark.parametrize("pair", [False, True])
def test_debug_variant_parity(debug_lib, B, H, N, d, causal, pair):
    if pair and d != 128:
        pytest.skip("the CTA-pair backward is built for d = 128")
    w = W.Workload("dbg", B, H, N, d, causal, seed=7100 + N + d)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=causal, scale=w.scale)
    A.fattn_set_bwd_pair(pair)
    try:
        dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    finally:
        A.fattn_set_bwd_pair(False)
    status = A.fattn_check_status()
    assert status == 0, _lib.status_string(status)
    o_ref, l_ref = oracle.attention_forward(inp["q"], inp["k"], inp["v"], causal, w.scale)
    check_o(to_np(o), o_ref, "O (debug)")
    check_l(to_np(lse), l_ref, "L (debug)")
    gq, gk, gv, _ = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], causal,
                                              w.scale)
    check_grad(to_np(dq), gq, "dQ (debug)")
    check_grad(to_np(dk), gk, "dK (debug)")
    check_grad(to_np(dv), gv, "dV (debug)")


def test_debug_variant_fp8_forward(debug_lib):
    w = W.Workload("dbg8", 1, 2, 500, 128, True, backward=False, seed=7300)
    inp = W.make_inputs(w)
    q8, sq = A.fattn_quantize_fp8(inp["q"].cuda())
    k8, sk = A.fattn_quantize_fp8(inp["k"].cuda())
    v8t, sv = A.fattn_quantize_fp8(inp["v"].cuda(), transposed=True)
    o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=True, scale=w.scale)
    status = A.fattn_check_status()
    assert status == 0, _lib.status_string(status)
    o_ref, l_ref = oracle.attention_fp8_reference(q8.cpu().numpy(), sq.cpu().numpy(),
                                                  k8.cpu().numpy(), sk.cpu().numpy(),
                                                  v8t.cpu().numpy(), sv.cpu().numpy(), True,
                                                  w.scale)
    check_l(to_np(lse), l_ref, "L(fp8, debug)")
    assert torch.isfinite(o.float()).all()
