"""Timeout path of the bounded waits, exercised without faulting the GPU:
a kernel waits on a barrier nothing completes, gives up after a short
budget and records FATTN_ERR_TIMEOUT; the context stays usable."""

import pytest
import torch

from exact_attention_fattn_gb300 import _lib
from exact_attention_fattn_gb300 import attention as A

pytestmark = pytest.mark.gpu


def test_selftest_timeout_reports_and_clears():
    assert A.fattn_check_status() == 0
    assert A.fattn_selftest_timeout(2_000_000) == _lib.FATTN_OK
    assert A.fattn_check_status() == _lib.FATTN_ERR_TIMEOUT
    assert A.fattn_check_status() == _lib.FATTN_OK          # cleared
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0                       # context still usable


def test_wait_budget_knob_roundtrip():
    A.fattn_set_wait_budget(1 << 30)
    A.fattn_set_wait_budget(0)          # back to the default
    assert A.fattn_check_status() == 0


def test_binding_refuses_mismatched_buffers():
    """Caller-provided buffers of the wrong shape, dtype or device are refused
    before anything is launched (the kernels would write past them)."""
    q = torch.zeros((1, 2, 256, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        A.fattn_fwd(q, q, q, out=torch.empty((1, 2, 255, 128), dtype=torch.bfloat16,
                                             device="cuda"))
    with pytest.raises(ValueError):
        A.fattn_fwd(q, q, q, lse=torch.empty((1, 2, 256), dtype=torch.float32))
    o, lse = A.fattn_fwd(q, q, q)
    with pytest.raises(ValueError):
        A.fattn_bwd(q, q, q, o, q, lse, dq=torch.empty_like(q, dtype=torch.float32))
    with pytest.raises(ValueError):
        A.fattn_bwd(q, q, q, o, q, lse, workspace=torch.empty(16, dtype=torch.float32,
                                                              device="cuda"))
    with pytest.raises(TypeError):
        A.fattn_quantize_fp8(q, signs=torch.ones(128, dtype=torch.float32))
    q8, sq = A.fattn_quantize_fp8(q)
    v8t, sv = A.fattn_quantize_fp8(q, transposed=True)
    with pytest.raises(ValueError):
        A.fattn_fwd_fp8(q8, sq.cpu(), q8, sq, v8t, sv)
    with pytest.raises(ValueError):
        A.fattn_fwd_fp8(q8, sq[:, :, :1].contiguous(), q8, sq, v8t, sv)
    assert A.fattn_check_status() == 0
