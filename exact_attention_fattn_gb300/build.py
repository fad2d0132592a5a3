"""Build libfattn.so in-tree with nvcc (sm_103a only).

The translation units are compiled in parallel and linked into one shared
library that exports the C ABI of include/fattn.h.  No PyTorch headers are
involved: the library is plain CUDA C++.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libfattn.so")
BUILD_DIR = os.path.join(PKG, "_build")
# Debug variant for tests: every kernel range-checks its computed shared-
# memory, TMEM and global indices (a failed check is reported as
# FATTN_ERR_DEBUG_CHECK, not a trap), and the forward's K/V ring has its
# minimum depth of two stages, so that the ring phases wrap as often as
# they can.
DEBUG_LIB_PATH = os.path.join(PKG, "libfattn_debug.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_FLAGS = ["-DFATTN_DEBUG", "-DFATTN_FWD_STAGES=2"]
SOURCES = ["fattn_api.cu", "fattn_fwd.cu", "fattn_bwd.cu", "fattn_bwd2.cu", "fattn_bwd_aux.cu",
           "fattn_fp8.cu", "fattn_sched.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libfattn")
    return cand


def _inputs_newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False,
          debug: bool = False) -> str:
    """Compile every .cu into libfattn.so next to this file (with debug=True:
    libfattn_debug.so, the checked variant); returns its path."""
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    extra = DEBUG_FLAGS if debug else []
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "fattn.h"))
    objs, jobs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _inputs_newer(obj, [path] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", path, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _inputs_newer(lib_path, objs):
        tmp = lib_path + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
