"""FP8 forward ("FlashAttention v1～v4" v3 §3): block quantization on the GPU
bit for bit against the oracle's, and the FP8 forward against the exact
attention of the dequantized inputs within the e4m3 bound."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import to_np
from tolerances import check_l, check_o_fp8

pytestmark = pytest.mark.gpu


def _quantize_all(inp):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    q8, sq = A.fattn_quantize_fp8(q)
    k8, sk = A.fattn_quantize_fp8(k)
    v8t, sv = A.fattn_quantize_fp8(v, transposed=True)
    assert A.fattn_check_status() == 0
    return q8, sq, k8, sk, v8t, sv


@pytest.mark.parametrize("B,H,N,outliers", [
    (1, 2, 300, False), (2, 3, 128, False), (1, 1, 1, False), (1, 2, 1000, True),
])
def test_quantize_bit_exact(B, H, N, outliers):
    w = W.Workload("q8", B, H, N, 128, False, seed=900 + N,
                   outlier_frac=0.01 if outliers else 0.0, outlier_mult=20.0)
    inp = W.make_inputs(w, with_grad=False)
    if N >= 256:
        inp["k"][0, 0, 128:256] = 0          # an all-zero block
    q8, sq, k8, sk, v8t, sv = _quantize_all(inp)
    for name, codes, scales, tr in (("q", q8, sq, False), ("k", k8, sk, False), ("v", v8t, sv, True)):
        want_c, want_s = oracle.block_quantize(inp[name], transpose=tr)
        assert np.array_equal(codes.cpu().numpy(), want_c), f"{name} codes differ"
        assert np.array_equal(scales.cpu().numpy(), want_s), f"{name} scales differ"


@pytest.mark.parametrize("B,H,N,causal,outliers", [
    (1, 2, 256, False, False),
    (1, 2, 300, True, False),
    (2, 2, 640, True, True),
    (1, 1, 1, False, False),
    (1, 3, 1000, False, False),
])
def test_fwd_fp8_matches_reference(B, H, N, causal, outliers):
    w = W.Workload("f8", B, H, N, 128, causal, seed=950 + N,
                   outlier_frac=0.01 if outliers else 0.0, outlier_mult=20.0)
    inp = W.make_inputs(w, with_grad=False)
    q8, sq, k8, sk, v8t, sv = _quantize_all(inp)
    o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=causal, scale=w.scale)
    assert A.fattn_check_status() == 0
    o_ref, l_ref = oracle.attention_fp8_reference(q8.cpu().numpy(), sq.cpu().numpy(),
                                                  k8.cpu().numpy(), sk.cpu().numpy(),
                                                  v8t.cpu().numpy(), sv.cpu().numpy(),
                                                  causal, w.scale)
    v_deq = oracle.block_dequantize(v8t.cpu().numpy(), sv.cpu().numpy(), N, transposed=True)
    check_o_fp8(to_np(o), o_ref, float(np.abs(v_deq).max()))
    check_l(to_np(lse), l_ref)


@pytest.mark.parametrize("tau", [0.0, 16.0])
def test_fwd_fp8_rescale_threshold(tau):
    """Any rescale threshold gives the FP8 result: the FP8 forward clamps it
    at 8, because its e4m3 probabilities (up to 2^tau) saturate at 448."""
    w = W.Workload("f8tau", 1, 2, 700, 128, True, outlier_frac=0.05, outlier_mult=20.0,
                   backward=False, seed=98)
    inp = W.make_inputs(w)
    q8, sq, k8, sk, v8t, sv = _quantize_all(inp)
    A.fattn_set_rescale_threshold(tau)
    try:
        o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=True, scale=w.scale)
        assert A.fattn_check_status() == 0
    finally:
        A.fattn_set_rescale_threshold(-1.0)
    o_ref, l_ref = oracle.attention_fp8_reference(q8.cpu().numpy(), sq.cpu().numpy(),
                                                  k8.cpu().numpy(), sk.cpu().numpy(),
                                                  v8t.cpu().numpy(), sv.cpu().numpy(),
                                                  True, w.scale)
    v_deq = oracle.block_dequantize(v8t.cpu().numpy(), sv.cpu().numpy(), w.N, transposed=True)
    check_o_fp8(to_np(o), o_ref, float(np.abs(v_deq).max()))
    check_l(to_np(lse), l_ref)


def test_fp8_rejects_d64():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        A.fattn_quantize_fp8(q)


# Incoherent processing ("FlashAttention v1～v4" v3 §3): Q and K rotated by
# the same random orthogonal matrix diag(s) H / sqrt(d) before quantization.

ENTRY_OUTLIERS = W.Workload("f8_entry_outliers", 1, 4, 1000, 128, False, backward=False,
                            seed=960, entry_outlier_frac=0.01, entry_outlier_std=10.0)


@pytest.mark.parametrize("B,H,N,outliers", [
    (1, 2, 300, False), (2, 1, 128, False), (1, 1, 1, False), (1, 2, 1000, True),
])
def test_quantize_rotated_bit_exact(B, H, N, outliers):
    w = W.Workload("q8r", B, H, N, 128, False, seed=970 + N, backward=False,
                   entry_outlier_frac=0.01 if outliers else 0.0, entry_outlier_std=10.0)
    inp = W.make_inputs(w)
    if N >= 256:
        inp["q"][0, 0, 128:256] = 0          # an all-zero block stays zero with scale 1
    signs = W.random_signs(128, seed=N)
    for name in ("q", "k"):
        codes, scales = A.fattn_quantize_fp8(inp[name].cuda(), signs=signs.cuda())
        assert A.fattn_check_status() == 0
        want_c, want_s = oracle.block_quantize(inp[name], signs=signs.numpy())
        assert np.array_equal(codes.cpu().numpy(), want_c), f"{name} codes differ"
        assert np.array_equal(scales.cpu().numpy(), want_s), f"{name} scales differ"


def _fwd_fp8_rotated(inp, w, signs):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    s = None if signs is None else signs.cuda()
    q8, sq = A.fattn_quantize_fp8(q, signs=s)
    k8, sk = A.fattn_quantize_fp8(k, signs=s)
    v8t, sv = A.fattn_quantize_fp8(v, transposed=True)
    o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=w.causal, scale=w.scale)
    assert A.fattn_check_status() == 0
    return (q8, sq, k8, sk, v8t, sv), to_np(o), to_np(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_fp8_rotated_matches_reference(causal):
    """The forward on rotated codes is the same kernel on other inputs: it
    matches the exact attention of the dequantized rotated Q, K and V."""
    w = W.Workload("f8r", 1, 2, 640, 128, causal, backward=False, seed=980,
                   entry_outlier_frac=0.01, entry_outlier_std=10.0)
    inp = W.make_inputs(w)
    codes, o, lse = _fwd_fp8_rotated(inp, w, W.random_signs(128, seed=3))
    o_ref, l_ref = oracle.attention_fp8_reference(*(c.cpu().numpy() for c in codes), causal,
                                                  w.scale)
    v_deq = oracle.block_dequantize(codes[4].cpu().numpy(), codes[5].cpu().numpy(), w.N,
                                    transposed=True)
    check_o_fp8(o, o_ref, float(np.abs(v_deq).max()))
    check_l(lse, l_ref)


def test_rotation_lowers_fp8_error_on_entry_outliers():
    """Against the exact attention of the bf16 inputs, rotating Q and K
    before block quantization lowers the FP8 forward's RMS error on inputs
    with isolated large entries (measured ratio about 2 on this workload)."""
    w = ENTRY_OUTLIERS
    inp = W.make_inputs(w)
    o_exact, l_exact = oracle.attention_forward(inp["q"], inp["k"], inp["v"], w.causal, w.scale)
    _, o_plain, l_plain = _fwd_fp8_rotated(inp, w, None)
    _, o_rot, l_rot = _fwd_fp8_rotated(inp, w, W.random_signs(128, seed=11))
    err_plain = float(np.sqrt(np.mean((o_plain - o_exact) ** 2)))
    err_rot = float(np.sqrt(np.mean((o_rot - o_exact) ** 2)))
    assert err_rot < 0.75 * err_plain, (err_rot, err_plain)
    lerr_plain = float(np.abs(l_plain - l_exact).max())
    lerr_rot = float(np.abs(l_rot - l_exact).max())
    assert lerr_rot < lerr_plain, (lerr_rot, lerr_plain)


def test_rotated_quantize_rejects_transposed_and_d64():
    s = torch.ones(128, dtype=torch.float32, device="cuda")
    x = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        A.fattn_quantize_fp8(x, transposed=True, signs=s)
    x64 = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        A.fattn_quantize_fp8(x64, signs=torch.ones(64, dtype=torch.float32, device="cuda"))


def test_fwd_fp8_tiny_value_block():
    """One V block about 1e-35 of the others: its block-scale ratio rho is far
    below 2^-100, where the forward clamps log2(rho).  The output stays finite
    and matches the exact attention of the dequantized inputs within the FP8
    bound (that block's contribution rounds to e4m3 zero either way), and L
    is unaffected (the row sums still count its probabilities)."""
    w = W.Workload("f8tiny", 1, 2, 512, 128, False, backward=False, seed=991)
    inp = W.make_inputs(w)
    inp["v"][:, :, 128:256] = (inp["v"][:, :, 128:256].float() * 1e-35).to(torch.bfloat16)
    q8, sq, k8, sk, v8t, sv = _quantize_all(inp)
    assert float(sv[0, 0, 1]) / float(sv.max()) < 2.0 ** -100
    o, lse = A.fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal=False, scale=w.scale)
    assert A.fattn_check_status() == 0
    o_np, l_np = to_np(o), to_np(lse)
    assert np.isfinite(o_np).all() and np.isfinite(l_np).all()
    o_ref, l_ref = oracle.attention_fp8_reference(q8.cpu().numpy(), sq.cpu().numpy(),
                                                  k8.cpu().numpy(), sk.cpu().numpy(),
                                                  v8t.cpu().numpy(), sv.cpu().numpy(),
                                                  False, w.scale)
    v_deq = oracle.block_dequantize(v8t.cpu().numpy(), sv.cpu().numpy(), w.N, transposed=True)
    check_o_fp8(o_np, o_ref, float(np.abs(v_deq).max()))
    check_l(l_np, l_ref)
