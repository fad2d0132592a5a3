"""FP8 (e4m3) block quantization and the attention it feeds.

TEST INFRASTRUCTURE ONLY (see the package docstring): it shares no code with
the CUDA library.

"FlashAttention v1～v4" v3 §3 quantizes Q, K and V to FP8 with one scale per
computation block (block quantization) instead of one per tensor.  The pages
fix neither the 8-bit encoding nor the block shape nor the rounding; the
reading taken here:

* format e4m3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
  infinities; codes 0x7F / 0xFF are NaN; largest finite value 1.75 * 2^8 = 448;
  exponent field 0 holds the subnormals m * 2^-9;
* a block is 128 consecutive rows of one (batch, head) with all d columns
  (the kernels' tile);
* scale = amax(|x| over the block) / 448, rounded to fp32 (1 for an all-zero
  block); code = e4m3(x * (1 / scale)), the reciprocal and the product each
  rounded to fp32, then rounded to nearest e4m3 (ties to an even code) and
  saturated to +-448.  These steps decide an integer, so they are taken in
  fp32 as the kernel takes them;
* the value a code stands for is decode(code) * scale (exact in fp64);
* incoherent processing (v3 §3: Q and K multiplied by one random orthogonal
  matrix M before quantization, QM (KM)^T = Q K^T) uses the randomized
  Hadamard transform M = diag(s) H / sqrt(d), H the Sylvester-Hadamard matrix
  and s a caller-given vector of +-1 signs.  It is applied row by row in fp32
  as the kernel applies it -- the signs, then the butterflies (a + b, a - b)
  at strides 1, 2, 4, ..., d/2, then one multiplication by fp32(1/sqrt(d)) --
  because its roundings decide the codes.

``attention_fp8_reference`` is the exact attention of the dequantized inputs
(the plain definition, via ``attention_forward``): what an FP8 forward
computes up to the rounding of its probabilities to e4m3.
"""

from __future__ import annotations

import numpy as np

from .attention import attention_forward, to_f64

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def _e4m3_table() -> np.ndarray:
    """Value of every non-negative code 0x00..0x7E, from its bit fields."""
    vals = np.empty(0x7F, dtype=np.float64)
    for code in range(0x7F):
        e, m = (code >> 3) & 0xF, code & 0x7
        vals[code] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()   # increasing in the code


def e4m3_decode(codes) -> np.ndarray:
    """fp64 value of uint8 e4m3 codes (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, E4M3_VALUES[np.minimum(mag, 0x7E)])
    return np.where(c & 0x80, -out, out)


def e4m3_encode(x) -> np.ndarray:
    """Round fp32 values to the nearest e4m3 code, ties to the even code,
    saturating at +-448 (NaN -> 0x7F)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    hi = np.searchsorted(E4M3_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = E4M3_VALUES[hi] - a
    d_lo = a - E4M3_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)                   # saturation
    code = np.where(np.isnan(x), 0x7F, code)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


def hadamard_rotate_fp32(x, signs) -> np.ndarray:
    """x [..., d] (d a power of two) times diag(signs) H / sqrt(d), in fp32,
    one rounding per butterfly, strides 1, 2, ..., d/2 in that order."""
    y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = y.shape[-1]
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a, b = z[..., 0, :], z[..., 1, :]
        y = np.stack([(a + b).astype(np.float32), (a - b).astype(np.float32)],
                     axis=-2).reshape(y.shape)
        h *= 2
    return (y * np.float32(1.0 / np.sqrt(d))).astype(np.float32)


def block_quantize(x, transpose: bool = False, signs=None):
    """Quantize a [B, H, N, d] tensor block by block (128 rows of a head),
    after the randomized Hadamard rotation when ``signs`` is given.

    Returns (codes, scales): codes uint8 [B, H, N, d], or [B, H, d, Np] with Np
    = N rounded up to 128 and zero codes past N when ``transpose``; scales
    fp32 [B, H, ceil(N / 128)].
    """
    xf = np.asarray(to_f64(x), dtype=np.float32)
    if signs is not None:
        xf = hadamard_rotate_fp32(xf, signs)
    B, H, N, d = xf.shape
    nt = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    scales = np.empty((B, H, nt), dtype=np.float32)
    codes = np.zeros((B, H, N, d), dtype=np.uint8)
    for t in range(nt):
        blk = xf[:, :, t * BLOCK_ROWS:(t + 1) * BLOCK_ROWS, :]
        amax = np.abs(blk).max(axis=(2, 3)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        inv = (np.float32(1.0) / s).astype(np.float32)
        scales[:, :, t] = s
        codes[:, :, t * BLOCK_ROWS:(t + 1) * BLOCK_ROWS, :] = e4m3_encode(
            (blk * inv[:, :, None, None]).astype(np.float32))
    if transpose:
        np_ = nt * BLOCK_ROWS
        out = np.zeros((B, H, d, np_), dtype=np.uint8)
        out[:, :, :, :N] = codes.transpose(0, 1, 3, 2)
        return out, scales
    return codes, scales


def block_dequantize(codes, scales, N: int, transposed: bool = False) -> np.ndarray:
    """fp64 [B, H, N, d] values of block-quantized codes."""
    c = np.asarray(codes)
    if transposed:
        c = c[:, :, :, :N].transpose(0, 1, 3, 2)
    vals = e4m3_decode(c)
    s = np.repeat(np.asarray(scales, dtype=np.float64), BLOCK_ROWS, axis=2)[:, :, :N]
    return vals * s[:, :, :, None]


def attention_fp8_reference(q8, sq, k8, sk, v8t, sv, causal: bool, scale: float):
    """Exact fp64 attention (O, L) of the dequantized FP8 inputs; v8t is the
    transposed [B, H, d, Np] layout."""
    N = np.asarray(q8).shape[2]
    q = block_dequantize(q8, sq, N)
    k = block_dequantize(k8, sk, N)
    v = block_dequantize(v8t, sv, N, transposed=True)
    return attention_forward(q, k, v, causal, scale)
