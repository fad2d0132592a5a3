"""The microbenchmarks' host-side pieces (no GPU needed).

exp2_rate.cu hard-codes the cubic it times; these constants must be the
near-minimax relative-error fit of 2^f on [-1/2, 1/2] that run.py derives,
and that fit must meet the error the design notes quote.
"""

import os
import re

import numpy as np

from exact_attention_fattn_gb300.microbench import run as mb


def _constants():
    src = open(os.path.join(mb.HERE, "exp2_rate.cu")).read()
    vals = {}
    for name in ("kC0", "kC1", "kC2", "kC3"):
        m = re.search(rf"constexpr float {name} = ([0-9.eE+-]+)f;", src)
        assert m, name
        vals[name] = float(m.group(1))
    return np.array([vals["kC0"], vals["kC1"], vals["kC2"], vals["kC3"]])


def test_exp2_cubic_matches_fit():
    c, err = mb.fit_exp2_cubic()
    assert err < 7.6e-5
    np.testing.assert_allclose(_constants(), c, rtol=0, atol=2e-7)


def test_exp2_cubic_error_in_fp32():
    # fp32 Horner with a single rounding per step, as the fused multiply-adds do
    c = _constants().astype(np.float32)
    f = np.linspace(-0.5, 0.5, 100001).astype(np.float32)
    p = np.float32(c[3])
    for k in (2, 1, 0):
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c[k])).astype(np.float32)
    rel = np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)
    assert rel.max() < 7.6e-5
    # 2^(n + f) = 2^n * p(f): the exponent-field step is exact, so the whole
    # range inherits the same bound (checked at a few integer shifts)
    for n in (-100, -10, 0, 3):
        y = np.ldexp(p.astype(np.float64), n)
        assert (np.abs(y / np.exp2(f.astype(np.float64) + n) - 1.0)).max() < 7.6e-5


def test_microbench_sources_compile(tmp_path):
    """Every committed microbenchmark compiles for sm_103a (object only; no GPU)."""
    import shutil
    import subprocess

    import pytest

    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc"
                                    if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    for name, src in mb.PROGRAMS.items():
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
               "--expt-relaxed-constexpr", "-c", os.path.join(mb.HERE, src),
               "-o", str(tmp_path / (name + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, f"{src}: {r.stderr[-2000:]}"
