"""The checked debug variant of the library (FATTN_DEBUG: every kernel
range-checks its computed shared-memory, TMEM and global indices and reports
a failed check as FATTN_ERR_DEBUG_CHECK instead of trapping; the forward's
K/V ring at its minimum depth of two stages) builds and exports the same C
ABI.  Its GPU run is in test_debug_build_gpu.py."""

import ctypes

from exact_attention_fattn_gb300 import _lib, build
from test_abi import declared_functions


def test_debug_variant_builds_and_exports_the_abi():
    path = build.build(debug=True)
    assert path.endswith("libfattn_debug.so")
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    lib.fattn_status_string.restype = ctypes.c_char_p
    assert b"debug" in lib.fattn_status_string(_lib.FATTN_ERR_DEBUG_CHECK)
