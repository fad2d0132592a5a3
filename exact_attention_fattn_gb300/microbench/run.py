"""Build and run the GB300 microbenchmarks behind the kernel design choices.

    python -m exact_attention_fattn_gb300.microbench.run [mma|reduce|exp2|load|fit ...]

`mma`, `reduce`, `exp2` and `load` compile the matching .cu file for sm_103a
into _build/ next to this file and run it on the current GPU; `fit` (CPU only)
prints the cubic for 2^f on [-1/2, 1/2] whose coefficients exp2_rate.cu uses.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
PROGRAMS = {"mma": "mma_rate.cu", "reduce": "reduce_rate.cu", "exp2": "exp2_rate.cu",
            "load": "load_rate.cu"}
# extra link flags (load_rate.cu encodes tensor maps through the driver API)
LINK = {"load": ["-lcuda"]}


def fit_exp2_cubic(iters: int = 200):
    """Near-minimax relative-error cubic for 2^f on [-1/2, 1/2].

    Lawson's iteration: weighted least squares whose weights are multiplied
    by the current absolute relative error each round, which converges to
    the equioscillating (minimax) solution.
    """
    import numpy as np

    f = np.linspace(-0.5, 0.5, 20001)
    y = 2.0 ** f
    V = np.vander(f, 4, increasing=True)
    w = np.ones_like(f)
    for _ in range(iters):
        A = V / y[:, None] * np.sqrt(w)[:, None]
        c, *_ = np.linalg.lstsq(A, np.sqrt(w), rcond=None)
        err = np.abs(V @ c / y - 1.0)
        w = w * err
        w /= w.sum()
    return c, float(np.abs(V @ c / y - 1.0).max())


def build(name: str) -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(HERE, PROGRAMS[name])
    exe = os.path.join(BUILD, name + "_rate")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "--expt-relaxed-constexpr", src, "-o", exe] + LINK.get(name, [])
    subprocess.run(cmd, check=True)
    return exe


def main(argv: list[str]) -> int:
    names = argv or ["fit", "mma", "reduce", "exp2", "load"]
    for name in names:
        print(f"== {name}", flush=True)
        if name == "fit":
            c, err = fit_exp2_cubic()
            print("c0..c3 =", ", ".join(f"{v:.9g}" for v in c), f"; max relative error {err:.3e}")
            continue
        rc = subprocess.run([build(name)]).returncode
        if rc != 0:
            return rc
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
