"""Parity tolerances (GPU result vs the fp64 oracle) and their checks.

The bounds are the ones stated for this path:
  O      : max |err| <= 1e-2 and mean |err| <= 1e-3
  L      : max |err| <= 1e-3
  dQ/dK/dV: max |err| <= 5e-2 * max |reference|   (per tensor)
One reading is applied to O: an element whose reference magnitude is >= 4
has a bf16 spacing of 2^-5 or more, so merely storing the exact value as
bf16 can miss it by more than 1e-2; such an element may differ by up to one
bf16 spacing of its reference value instead.
"""

import numpy as np

O_MAX, O_MEAN, L_MAX, GRAD_REL = 1e-2, 1e-3, 1e-3, 5e-2


def bf16_spacing(x):
    """Distance between adjacent bf16 values around |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_o(o_gpu, o_ref, what="O"):
    err = np.abs(o_gpu - o_ref)
    allow = np.maximum(O_MAX, bf16_spacing(o_ref))
    worst = float((err - allow).max())
    assert worst <= 0, f"{what}: max err {err.max():.3e} exceeds its bound (by {worst:.3e})"
    assert err.mean() <= O_MEAN, f"{what}: mean err {err.mean():.3e} > {O_MEAN}"
    return float(err.max()), float(err.mean())


def check_l(l_gpu, l_ref, what="L"):
    err = np.abs(l_gpu - l_ref)
    assert np.isfinite(l_gpu).all(), f"{what}: non-finite values"
    assert err.max() <= L_MAX, f"{what}: max err {err.max():.3e} > {L_MAX}"
    return float(err.max())


GRAD_FLOOR = 1e-4


def check_grad(g_gpu, g_ref, what):
    # The bound is relative to max |reference|.  When the exact gradient is
    # (close to) zero everywhere -- e.g. dQ and dK at N = 1, where the
    # softmax of a single score is constant -- the scale is floored at 1e-4
    # so that fp32 rounding noise is not judged against zero.
    ref_max = max(float(np.abs(g_ref).max()), GRAD_FLOOR)
    err = float(np.abs(g_gpu - g_ref).max())
    assert np.isfinite(g_gpu).all(), f"{what}: non-finite values"
    assert err <= GRAD_REL * ref_max, f"{what}: max err {err:.3e} > {GRAD_REL} * {ref_max:.3e}"
    return err / max(ref_max, 1e-30)


# FP8 forward (e4m3 probabilities in P V): against the exact attention of the
# dequantized inputs.  Every probability that meets V is rounded to e4m3 (3
# mantissa bits, relative error <= 2^-4 with round to nearest); the row sum
# that normalises O is taken on the unrounded values, so
#   |O_fp8 - O_ref| <= 2^-4 * sum_k P_k |v_k| / l <= 2^-4 * max |V|
# per element (subnormal codes, below 2^-6, err by at most 2^-10 absolute
# each, far below this once weighted by P / l), plus the bf16 spacing of the
# stored output.  With independent rounding errors the typical error is
# ~2^-4 / sqrt(3) / sqrt(N_eff) * |V| (N_eff = keys that carry the row's
# weight); the mean bound below, 1 % of max |V|, leaves a wide margin for rows
# that few keys dominate.  L uses the fp32 probabilities and exact e4m3
# products in S: the bf16 path's bound applies.
FP8_O_MAX_REL, FP8_O_MEAN_REL = 2.0 ** -4, 1e-2


def check_o_fp8(o_gpu, o_ref, v_absmax, what="O(fp8)"):
    err = np.abs(o_gpu - o_ref)
    allow = FP8_O_MAX_REL * v_absmax + bf16_spacing(o_ref)
    worst = float((err - allow).max())
    assert worst <= 0, f"{what}: max err {err.max():.3e} exceeds its bound (by {worst:.3e})"
    assert err.mean() <= FP8_O_MEAN_REL * v_absmax, (
        f"{what}: mean err {err.mean():.3e} > {FP8_O_MEAN_REL} * max|V| = {FP8_O_MEAN_REL * v_absmax:.3e}")
    return float(err.max()), float(err.mean())
