"""Pins of the oracle's FP8 part (CPU only): the e4m3 format from its
definition, round-to-nearest-even with saturation, block quantization, and
plausible mistakes planted in a copy of the module that these pins catch.

The format facts come from the definition of e4m3 (1 sign, 4 exponent bits
with bias 7, 3 mantissa bits, no infinities, 0x7F NaN, largest finite 448),
written out here by hand, not computed by the module under test.
"""

import inspect
import types

import numpy as np
import pytest

import oracle.fp8 as fp8

# (code, value) written out from the bit fields by hand
KNOWN = [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x02, 2.0 ** -8), (0x07, 7 * 2.0 ** -9),   # subnormals
    (0x08, 2.0 ** -6), (0x09, 1.125 * 2.0 ** -6),                              # smallest normals
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x44, 3.0),
    (0x77, 240.0), (0x78, 256.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9)),
]


def check_known_codes(m):
    for code, val in KNOWN:
        assert m.e4m3_decode([code])[0] == val, hex(code)
        assert int(m.e4m3_encode(np.float32(val))) == code, (val, hex(code))
    assert np.isnan(m.e4m3_decode([0x7F])[0]) and np.isnan(m.e4m3_decode([0xFF])[0])


def check_table_monotone_and_round_trip(m):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = m.e4m3_decode(codes)
    pos = vals[: 0x7F]
    assert np.all(np.diff(pos) > 0) and pos[0] == 0.0 and pos[-1] == 448.0
    back = m.e4m3_encode(vals.astype(np.float32))
    same = (back == codes) | ((codes == 0x80) & (back == 0x80))
    assert np.all(same)


def check_ties_to_even(m):
    pos = m.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2          # exactly representable in fp32
    got = m.e4m3_encode(mids.astype(np.float32)).astype(int)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want)


def check_nearest(m):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-8, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    got = m.e4m3_decode(m.e4m3_encode(x))
    table = np.concatenate([-m.e4m3_decode(np.arange(0x7F, dtype=np.uint8))[::-1],
                            m.e4m3_decode(np.arange(0x7F, dtype=np.uint8))])
    best = np.abs(table[None, :] - x[:, None].astype(np.float64)).min(axis=1)
    assert np.all(np.abs(got - x) == best)


def check_saturation(m):
    big = np.array([448.0, 464.0, 480.0, 1e6, np.inf, -500.0], dtype=np.float32)
    assert m.e4m3_encode(big).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert int(m.e4m3_encode(np.float32(np.nan))) & 0x7F == 0x7F


def check_block_quantize(m):
    rng = np.random.default_rng(5)
    B, H, N, d = 2, 3, 300, 64
    x = (rng.standard_normal((B, H, N, d)) * rng.uniform(0.1, 30, (B, H, 1, 1))).astype(np.float32)
    x[0, 1, 128:256] = 0.0                                  # an all-zero block
    codes, s = m.block_quantize(x)
    assert codes.shape == (B, H, N, d) and s.shape == (B, H, 3) and s.dtype == np.float32
    assert s[0, 1, 1] == 1.0 and np.all(codes[0, 1, 128:256] == 0)
    for b in range(B):
        for h in range(H):
            for t in range(3):
                blk = x[b, h, t * 128:(t + 1) * 128]
                amax = np.abs(blk).max()
                if amax == 0:
                    continue
                assert s[b, h, t] == np.float32(amax / np.float32(448.0))
                # the largest element lands on (or within one code of) +-448
                assert np.abs(m.e4m3_decode(codes[b, h, t * 128:(t + 1) * 128])).max() >= 416.0
    deq = m.block_dequantize(codes, s, N)
    sfull = np.repeat(s.astype(np.float64), 128, axis=2)[:, :, :N, None]
    err = np.abs(deq - x)
    assert np.all(err <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * sfull + 1e-12)
    ct, st = m.block_quantize(x, transpose=True)
    assert ct.shape == (B, H, d, 384) and np.array_equal(st, s)
    assert np.array_equal(ct[:, :, :, :N], codes.transpose(0, 1, 3, 2)) and np.all(ct[:, :, :, N:] == 0)


def check_reference_on_exact_inputs(m):
    """Inputs that block quantization represents exactly (block amax 448 * 2^k,
    entries e4m3 values * 2^k): the FP8 reference equals plain attention."""
    rng = np.random.default_rng(9)
    B, H, N, d = 1, 2, 200, 64
    pos = m.e4m3_decode(np.arange(0x7F, dtype=np.uint8))

    def exact(seed_shift):
        v = rng.choice(pos[40:110], size=(B, H, N, d)) * rng.choice([-1.0, 1.0], size=(B, H, N, d))
        v[:, :, ::128, 0] = 448.0                    # block amax exactly 448 in every block
        return (v * 2.0 ** seed_shift).astype(np.float32)

    q, k, v = exact(-9), exact(-8), exact(-7)
    q8, sq = m.block_quantize(q)
    k8, sk = m.block_quantize(k)
    v8t, sv = m.block_quantize(v, transpose=True)
    o_ref, l_ref = m.attention_forward(q.astype(np.float64), k.astype(np.float64),
                                       v.astype(np.float64), True, 0.125)
    o, l = m.attention_fp8_reference(q8, sq, k8, sk, v8t, sv, True, 0.125)
    assert np.array_equal(o, o_ref) and np.array_equal(l, l_ref)


def check_hadamard_basis_vectors(m):
    """e_k -> s_k times row k of the Sylvester-Hadamard matrix (entries
    (-1)^popcount(k & j)) over sqrt(d): every butterfly adds +-s_k to 0, so
    the only rounding is the final fp32 multiplication."""
    d = 128
    rng = np.random.default_rng(21)
    signs = rng.choice([-1.0, 1.0], d)
    c = np.float32(1.0 / np.sqrt(d))
    eye = np.eye(d, dtype=np.float32)
    y = m.hadamard_rotate_fp32(eye, signs)
    jj = np.arange(d)
    for k in range(d):
        parity = np.array([bin(k & j).count("1") & 1 for j in jj])
        want = (np.float32(signs[k]) * np.where(parity, -1.0, 1.0).astype(np.float32) * c)
        assert np.array_equal(y[k], want.astype(np.float32)), k


def check_hadamard_matches_matrix(m):
    """Random rows against the explicit product x diag(s) H / sqrt(d) in fp64
    (H built by Kronecker products), and dot products preserved."""
    d = 128
    rng = np.random.default_rng(22)
    signs = rng.choice([-1.0, 1.0], d)
    H = np.array([[1.0]])
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    x = (rng.standard_normal((64, d)) * 3).astype(np.float32)
    want = (x.astype(np.float64) * signs) @ H / np.sqrt(d)
    got = m.hadamard_rotate_fp32(x, signs).astype(np.float64)
    assert np.abs(got - want).max() <= 1e-5 * np.abs(want).max()
    q, k = x[:32], x[32:]
    dots = q.astype(np.float64) @ k.astype(np.float64).T
    dots_rot = got[:32] @ got[32:].T
    assert np.abs(dots_rot - dots).max() <= 1e-4 * np.abs(dots).max()
    # block_quantize with signs quantizes the rotated tensor
    xt = x.reshape(1, 1, 64, d)
    c1, s1 = m.block_quantize(xt, signs=signs)
    c2, s2 = m.block_quantize(m.hadamard_rotate_fp32(xt, signs))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


ALL_FP8_CHECKS = [check_known_codes, check_table_monotone_and_round_trip, check_ties_to_even,
                  check_nearest, check_saturation, check_block_quantize,
                  check_reference_on_exact_inputs, check_hadamard_basis_vectors,
                  check_hadamard_matches_matrix]


@pytest.mark.parametrize("check", ALL_FP8_CHECKS, ids=lambda c: c.__name__)
def test_fp8_pin(check):
    check(fp8)


MUTATIONS = {
    "exponent_bias_8": ("else (1.0 + m / 8.0) * 2.0 ** (e - 7)", "else (1.0 + m / 8.0) * 2.0 ** (e - 8)"),
    "subnormal_scale": ("m * 2.0 ** -9 if e == 0", "m * 2.0 ** -10 if e == 0"),
    "ties_away_from_zero": ("pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))",
                            "pick_hi = (d_hi <= d_lo)"),
    "truncation": ("pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))",
                   "pick_hi = d_hi == 0"),
    "overflow_to_nan": ("code = np.where(a >= E4M3_MAX, 0x7E, code)",
                        "code = np.where(a > E4M3_MAX, 0x7F, code)"),
    "scale_not_max": ("amax = np.abs(blk).max(axis=(2, 3)).astype(np.float32)",
                      "amax = np.abs(blk).mean(axis=(2, 3)).astype(np.float32)"),
    "scale_by_divide_not_multiply": ("(blk * inv[:, :, None, None]).astype(np.float32))",
                                     "(blk * s[:, :, None, None]).astype(np.float32))"),
    "transpose_forgotten": ("out[:, :, :, :N] = codes.transpose(0, 1, 3, 2)",
                            "out[:, :, :, :N] = codes.reshape(B, H, d, N)"),
    "dequant_drops_scale": ("return vals * s[:, :, :, None]", "return vals"),
    "hadamard_difference_swapped": ("(a - b).astype(np.float32)]", "(b - a).astype(np.float32)]"),
    "hadamard_no_normalisation": ("return (y * np.float32(1.0 / np.sqrt(d))).astype(np.float32)",
                                  "return y"),
    "hadamard_signs_ignored": ("y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)",
                               "y = np.asarray(x, dtype=np.float32)"),
    "hadamard_last_stage_skipped": ("    while h < d:", "    while h < d // 2:"),
}


def _mutant(old, new):
    src = inspect.getsource(fp8).replace("from .attention import", "from oracle.attention import")
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("oracle_fp8_mutant")
    exec(compile(src.replace(old, new), "<oracle_fp8_mutant>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_fp8_pins_catch_mutation(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for check in ALL_FP8_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except Exception:
            failed.append(check.__name__)
    assert failed, f"no pin caught mutation {name}"
