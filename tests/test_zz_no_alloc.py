"""fattn_bwd_noalloc, the backward pass for callers that cannot allocate
device memory at the point of the call (a plugin whose host framework owns
every allocation, a loop that cannot afford cudaMalloc's implicit
synchronisation, a caller without a spare buffer).  Its scratch is a fixed
array inside the library, so the call itself allocates nothing.

It must give what fattn_bwd gives with a caller-owned workspace, on every
call: the array keeps the previous call's contents, and a second call in a
row must not be affected by them.  This file is collected last on purpose.
"""

import pytest
import torch

from exact_attention_fattn_gb300 import _lib
from exact_attention_fattn_gb300 import attention as A
from exact_attention_fattn_gb300 import workloads as W
from gpu_util import to_np
from tolerances import check_grad

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, scale):
    B, H, N, d = q.shape
    return lib.fattn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, N, d, int(causal), scale,
                                 torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 333, 64, True), (2, 4, 1024, 128, False)])
def test_noalloc_matches_workspace_entry_point_twice(B, H, N, d, causal):
    lib = _lib.load()
    w = W.Workload("noalloc", B, H, N, d, causal, seed=2024 + N)
    inp = W.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = A.fattn_fwd(q, k, v, causal=causal, scale=w.scale)
    ref_dq, ref_dk, ref_dv = A.fattn_bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    assert A.fattn_check_status() == 0
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, w.scale)
        assert rc == _lib.FATTN_OK, _lib.status_string(rc)
        assert A.fattn_check_status() == 0
        check_grad(to_np(dq), to_np(ref_dq), "dQ")
        check_grad(to_np(dk), to_np(ref_dk), "dK")
        check_grad(to_np(dv), to_np(ref_dv), "dV")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, N, d = 1, 64, 4096, 128          # needs ~136 MB of scratch
    assert lib.fattn_bwd_workspace_bytes(B, H, N, d) > _lib.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = t.data_ptr()
    rc = lib.fattn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0, 0.088,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.FATTN_ERR_TOO_LARGE
    assert A.fattn_check_status() == 0
