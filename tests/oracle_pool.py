"""Run the fp64 oracle over many (batch, head) slices in parallel.

The full-size parity tests need the oracle on every head of a workload
(tens of seconds of fp64 work per workload).  Each head is an independent
problem, so the heads are spread over a pool of worker processes, one BLAS
thread each.  The pool is started with the ``spawn`` method: a process
forked from one that has already used the GPU can hang.

Only the tests use this module; it calls nothing but ``oracle``.
"""

from __future__ import annotations

import contextlib
import multiprocessing as mp
import os

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def workers() -> int:
    return max(1, len(os.sched_getaffinity(0)))


@contextlib.contextmanager
def pool():
    """A spawn-context pool whose workers each run a single BLAS thread."""
    saved = {k: os.environ.get(k) for k in _BLAS_VARS}
    for k in _BLAS_VARS:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        p = ctx.Pool(workers())
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield p
    finally:
        p.close()
        p.join()


# ---------------------------------------------------------------- jobs
# Each job takes CPU tensors of one head ([1, 1, N, d]) and returns numpy
# arrays for that head.

def head_forward(job):
    """O, L and A = sum_j P_ij |V_jc| (for the O tolerance) of one head."""
    import oracle

    q, k, v, causal, scale = job
    o, l = oracle.attention_forward(q, k, v, causal, scale)
    a = oracle.attention_abs_weighted_values(q, k, v, causal, scale)
    return o[0, 0], l[0, 0], a[0, 0]


def head_forward_backward(job):
    import oracle

    q, k, v, do, causal, scale = job
    o, l = oracle.attention_forward(q, k, v, causal, scale)
    a = oracle.attention_abs_weighted_values(q, k, v, causal, scale)
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, do, causal, scale)
    return o[0, 0], l[0, 0], dq[0, 0], dk[0, 0], dv[0, 0], a[0, 0]


def head_rows(job):
    """O, L, A, dQ on query rows ``qr`` and dK, dV on key rows ``kr`` of one head."""
    import oracle

    q, k, v, do, qr, kr, causal, scale = job
    o, l = oracle.attention_forward_rows(q, k, v, qr, causal, scale)
    a = oracle.attention_abs_weighted_values(q, k, v, causal, scale, rows=qr)
    dq = oracle.attention_backward_query_rows(q, k, v, do, qr, causal, scale)
    dk, dv = oracle.attention_backward_key_rows(q, k, v, do, kr, causal, scale)
    return o[0, 0], l[0, 0], dq[0, 0], dk[0, 0], dv[0, 0], a[0, 0]


def head_slice(inp, hflat, H, names):
    b, h = divmod(hflat, H)
    sl = (slice(b, b + 1), slice(h, h + 1))
    return tuple(inp[n][sl].clone() for n in names)
