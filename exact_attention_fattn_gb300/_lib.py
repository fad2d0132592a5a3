"""ctypes binding of libfattn (include/fattn.h): argument marshalling only.

Every computation runs in the CUDA kernels of libfattn.so.  If the library is
missing or cannot be loaded this module raises; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn.so")

FATTN_OK = 0
FATTN_ERR_INVALID_ARG = 1
FATTN_ERR_UNSUPPORTED = 2
FATTN_ERR_CUDA = 3
FATTN_ERR_TIMEOUT = 4
FATTN_ERR_TOO_LARGE = 5
FATTN_ERR_DEBUG_CHECK = 6
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); the order of argtypes follows include/fattn.h
SIGNATURES = {
    "fattn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                           _c_float, _vp]),
    "fattn_fp8_codes_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "fattn_quantize_fp8": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "fattn_quantize_fp8_rotated": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                            _vp]),
    "fattn_fwd_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                               _c_int, _c_int, _c_float, _vp]),
    "fattn_bwd_preprocess": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp]),
    "fattn_bwd_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "fattn_bwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_size,
                           _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp]),
    "fattn_bwd_prepare": (_c_int, [_vp, _vp, _vp, _vp, _c_size, _c_int, _c_int, _c_int, _c_int,
                                   _vp]),
    "fattn_bwd_main": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_size, _vp, _vp, _c_int, _c_int,
                                _c_int, _c_int, _c_int, _c_float, _vp]),
    "fattn_bwd_finish": (_c_int, [_vp, _c_size, _vp, _c_int, _c_int, _c_int, _c_int, _c_float,
                                  _vp]),
    "fattn_bwd_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_float, _vp]),
    "fattn_bwd_schedule": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    ctypes.c_longlong, _vp, _vp]),
    "fattn_bwd_schedule_items": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          ctypes.c_longlong, _vp, _vp]),
    "fattn_bwd_pair_schedule_items": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                               ctypes.c_longlong, _vp, _vp]),
    "fattn_check_status": (_c_int, [_vp]),
    "fattn_status_string": (ctypes.c_char_p, [_c_int]),
    "fattn_set_wait_budget": (None, [ctypes.c_longlong]),
    "fattn_set_rescale_threshold": (None, [_c_float]),
    "fattn_set_deterministic": (None, [ctypes.c_int]),
    "fattn_set_bwd_pair": (None, [ctypes.c_int]),
    "fattn_selftest_timeout": (_c_int, [ctypes.c_longlong, _vp]),
    "fattn_version": (ctypes.c_char_p, []),
}


class FattnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libfattn.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"libfattn.so not found at {p}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fattn_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != FATTN_OK:
        raise FattnError(fn, status, status_string(status))
