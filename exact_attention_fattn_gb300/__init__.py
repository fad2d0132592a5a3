"""libfattn: exact IO-aware attention on GB300 (sm_103a).

The compute lives in the CUDA library libfattn.so (C ABI in include/fattn.h);
this package holds its build script, a ctypes binding with the same entry
point names, and the seeded workload generator.
"""

from .attention import (  # noqa: F401
    default_scale,
    fattn_bwd,
    fattn_bwd_finish,
    fattn_bwd_main,
    fattn_bwd_prepare,
    fattn_bwd_schedule,
    fattn_bwd_schedule_items,
    fattn_bwd_pair_schedule_items,
    fattn_bwd_preprocess,
    fattn_bwd_workspace_bytes,
    fattn_check_status,
    fattn_fwd,
    fattn_fwd_fp8,
    fattn_quantize_fp8,
    fattn_selftest_timeout,
    fattn_set_bwd_pair,
    fattn_set_deterministic,
    fattn_set_rescale_threshold,
    fattn_set_wait_budget,
    workspace_for,
)
