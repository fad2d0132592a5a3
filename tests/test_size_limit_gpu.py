"""Parity at the size limit: tensors of just under 2^31 elements.

The library takes B*H*N*d < 2^31 (include/fattn.h).  These shapes sit 2^21
elements below that bound with a ragged N (1023: a partial last tile in every
head), so the last heads address O, dQ, dK, dV and the inputs at element
offsets close to 2^31 (byte offsets beyond 4 GiB for the bf16 tensors, 8 GiB
for the fp32 dQ accumulator).  The checked debug variant of the library runs
these shapes first.  Inputs are drawn on the GPU
(workloads.make_inputs_device); the fp64 oracle checks every element of O,
L, dQ, dK and dV on the first two and last two heads and on three seeded
heads in between, and the FP8 forward (quantization included) on the first
and last heads.
"""

import numpy as np
import pytest
import torch

import oracle
import oracle_pool as OP
from exact_attention_fattn_gb300 import _lib, build
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import to_np
from tolerances import check_grad, check_l, check_o, check_o_fp8

pytestmark = pytest.mark.gpu

LIMIT_SHAPES = [
    W.Workload("b128h128_n1023_d128", 128, 128, 1023, 128, False, seed=1007),
    W.Workload("b128h128_n1023_d128_causal", 128, 128, 1023, 128, True, seed=1008),
    W.Workload("b256h128_n1023_d64", 256, 128, 1023, 64, False, seed=1009),
]


def _heads(w):
    n = w.B * w.H
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 11)
    mid = torch.randperm(n - 4, generator=g)[:3] + 2
    return sorted({0, 1, n - 2, n - 1, *mid.tolist()})


def _slice(t, hf, H):
    b, h = divmod(hf, H)
    return t[b:b + 1, h:h + 1].cpu().clone()


@pytest.mark.parametrize("w", LIMIT_SHAPES[1:], ids=lambda w: w.name)
def test_size_limit_checked_variant(w):
    """First, the checked debug variant (every computed index range-checked,
    a failed check reported as a status instead of an access) at the same
    shapes, quantization and FP8 forward included: no check may fire, and
    the last head matches the oracle."""
    lib = _lib.load(build.build(debug=True))
    saved = _lib._lib
    _lib._lib = lib
    try:
        inp = W.make_inputs_device(w, "cuda")
        q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
        o, lse = A.fattn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        status = A.fattn_check_status()
        assert status == 0, _lib.status_string(status)
        if w.d == 128:
            q8, sq = A.fattn_quantize_fp8(q)
            k8, sk = A.fattn_quantize_fp8(k)
            v8t, sv = A.fattn_quantize_fp8(v, transposed=True)
            A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=w.causal, scale=w.scale)
            torch.cuda.synchronize()
            status = A.fattn_check_status()
            assert status == 0, _lib.status_string(status)
        hf = w.B * w.H - 1
        args = [_slice(inp[n], hf, w.H) for n in ("q", "k", "v", "do")]
        o_ref, l_ref = oracle.attention_forward(*args[:3], w.causal, w.scale)
        gq, gk, gv, _ = oracle.attention_backward(*args, w.causal, w.scale)
        check_o(to_np(_slice(o, hf, w.H)), o_ref, f"O (debug) last head of {w.name}")
        check_l(to_np(_slice(lse, hf, w.H)), l_ref, f"L (debug) last head of {w.name}")
        check_grad(to_np(_slice(dq, hf, w.H)), gq, "dQ (debug) last head")
        check_grad(to_np(_slice(dk, hf, w.H)), gk, "dK (debug) last head")
        check_grad(to_np(_slice(dv, hf, w.H)), gv, "dV (debug) last head")
    finally:
        _lib._lib = saved


@pytest.mark.parametrize("w", LIMIT_SHAPES, ids=lambda w: w.name)
def test_size_limit_fwd_bwd(w):
    assert w.B * w.H * w.N * w.d < 2 ** 31
    assert w.B * w.H * w.N * w.d > 2 ** 31 - 2 ** 22
    inp = W.make_inputs_device(w, "cuda")
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = A.fattn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert A.fattn_check_status() == 0
    heads = _heads(w)
    jobs = [tuple(_slice(inp[n], hf, w.H) for n in ("q", "k", "v", "do")) + (w.causal, w.scale)
            for hf in heads]
    got = [np.stack([to_np(_slice(t, hf, w.H))[0, 0] for hf in heads])
           for t in (o, lse, dq, dk, dv)]
    with OP.pool() as p:
        res = list(p.imap(OP.head_forward_backward, jobs))
    ref = [np.stack([r[i] for r in res]) for i in range(6)]
    tag = f"{w.name} heads {heads[0]}..{heads[-1]}"
    check_o(got[0], ref[0], f"O {tag}", abs_weighted=ref[5])
    check_l(got[1], ref[1], f"L {tag}")
    check_grad(got[2], ref[2], f"dQ {tag}")
    check_grad(got[3], ref[3], f"dK {tag}")
    check_grad(got[4], ref[4], f"dV {tag}")


def test_size_limit_fp8_forward():
    w = LIMIT_SHAPES[1]
    inp = W.make_inputs_device(w, "cuda", with_grad=False)
    q8, sq = A.fattn_quantize_fp8(inp["q"])
    k8, sk = A.fattn_quantize_fp8(inp["k"])
    v8t, sv = A.fattn_quantize_fp8(inp["v"], transposed=True)
    o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert A.fattn_check_status() == 0
    N = w.N
    for hf in (0, w.B * w.H - 1):
        # the codes and scales of this head, against the oracle's quantizer
        for name, codes, scales, tr in (("q", q8, sq, False), ("k", k8, sk, False),
                                        ("v", v8t, sv, True)):
            c_ref, s_ref = oracle.block_quantize(_slice(inp[name], hf, w.H), transpose=tr)
            assert np.array_equal(_slice(codes, hf, w.H).numpy(), c_ref), f"{name} codes, head {hf}"
            assert np.array_equal(_slice(scales, hf, w.H).numpy(), s_ref), f"{name} scales, head {hf}"
        qd = oracle.block_dequantize(_slice(q8, hf, w.H).numpy(), _slice(sq, hf, w.H).numpy(), N)
        kd = oracle.block_dequantize(_slice(k8, hf, w.H).numpy(), _slice(sk, hf, w.H).numpy(), N)
        vd = oracle.block_dequantize(_slice(v8t, hf, w.H).numpy(), _slice(sv, hf, w.H).numpy(), N,
                                     transposed=True)
        o_ref, l_ref = oracle.attention_forward(qd, kd, vd, True, w.scale)
        check_o_fp8(to_np(_slice(o, hf, w.H)), o_ref, float(np.abs(vd).max()),
                    f"O(fp8) head {hf}")
        check_l(to_np(_slice(lse, hf, w.H)), l_ref, f"L(fp8) head {hf}")
