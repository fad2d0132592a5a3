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
