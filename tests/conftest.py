import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfattn")


def _cuda_available():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """One line per parity check that ran: the errors against the oracle."""
    try:
        from tolerances import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    terminalreporter.section("parity against the fp64 oracle (max / mean abs error)")
    for test, what, fig in REPORT:
        extra = " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}"
                         for k, v in fig.items() if k not in ("max", "mean"))
        terminalreporter.write_line(
            f"{test.split('::')[-1]:<60} {what:<14} max {fig['max']:.3e}  "
            f"mean {fig['mean']:.3e}  {extra}")
