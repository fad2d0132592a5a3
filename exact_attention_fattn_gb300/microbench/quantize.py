"""Time the FP8 block quantization kernels through the library.

    python -m exact_attention_fattn_gb300.microbench.quantize [plain|tr|rot ...] [--n N]

Quantizes one bf16 [2, 32, N, 128] tensor of normal draws row-major
(``plain``, Q and K), transposed (``tr``, V) and after the Hadamard rotation
(``rot``), each timed from a CUDA graph of 20 launches, and prints the time
and the HBM rate (2 bytes read and 1 byte written per element).
"""

from __future__ import annotations

import argparse

import torch

from .. import attention as A


def time_mode(fn, reps: int = 20) -> float:
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    g.replay()
    a1.record()
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / reps * 1e3


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("modes", nargs="*", default=["plain", "tr", "rot"])
    ap.add_argument("--n", type=int, default=8192)
    args = ap.parse_args(argv)
    g = torch.Generator(device="cpu").manual_seed(7)
    x = torch.randn(2, 32, args.n, 128, generator=g).to(torch.bfloat16).cuda()
    signs = torch.ones(128, dtype=torch.float32, device="cuda")
    signs[1::2] = -1.0
    fns = {"plain": lambda: A.fattn_quantize_fp8(x),
           "tr": lambda: A.fattn_quantize_fp8(x, transposed=True),
           "rot": lambda: A.fattn_quantize_fp8(x, signs=signs)}
    for m in args.modes:
        us = time_mode(fns[m])
        print(f"{m:5s} N={args.n}: {us:7.1f} us  {x.numel() * 3 / us / 1e3:6.0f} GB/s", flush=True)
    rc = A.fattn_check_status()
    if rc != 0:
        raise RuntimeError(f"libfattn status {rc}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
