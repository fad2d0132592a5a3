"""The C ABI on the host (no GPU needed): the library loads, exports every
entry point that include/fattn.h declares, and rejects bad arguments before
it touches the device."""

import ctypes
import os
import re

import pytest

from exact_attention_fattn_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fattn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from exact_attention_fattn_gb300 import build

        build.build()
    return _lib.load()


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("fattn_fwd", "fattn_bwd", "fattn_bwd_preprocess", "fattn_bwd_workspace_bytes",
                 "fattn_check_status", "fattn_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fattn.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings_and_version(lib):
    assert lib.fattn_status_string(0) == b"ok"
    assert lib.fattn_status_string(4) == b"kernel wait timed out"
    assert lib.fattn_status_string(99) == b"unknown status"
    assert re.fullmatch(rb"\d+\.\d+\.\d+", lib.fattn_version())


def test_workspace_bytes(lib):
    def al(x):
        return (x + 255) // 256 * 256

    for B, H, N, d in ((1, 1, 1, 64), (2, 32, 4096, 128), (1, 16, 16384, 128), (3, 5, 77, 64)):
        rows = B * H * N
        np_ = (N + 127) // 128 * 128
        counters = al(4 * B * H * (np_ // 128))
        assert lib.fattn_bwd_workspace_bytes(B, H, N, d) == (2 * al(4 * B * H * np_)
                                                             + al(4 * rows * d) + counters)
    assert lib.fattn_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert lib.fattn_bwd_workspace_bytes(1, 1, 1, 96) == 0
    # the size limit: fewer than 2^31 elements per [B, H, N, d] tensor
    assert lib.fattn_bwd_workspace_bytes(1, 1, (1 << 24) - 1, 128) > 0
    assert lib.fattn_bwd_workspace_bytes(1, 1, 1 << 24, 128) == 0
    assert lib.fattn_bwd_workspace_bytes(2, 4, 1 << 21, 128) == 0
    assert lib.fattn_bwd_workspace_bytes(2, 4, (1 << 21) - 1, 128) > 0


GOOD = 0x10000  # a 16-byte aligned fake address; never dereferenced


@pytest.mark.parametrize("B,H,N,d,scale,ptr,want", [
    (0, 1, 128, 64, 0.125, GOOD, 1),
    (1, -1, 128, 64, 0.125, GOOD, 1),
    (1, 1, 0, 64, 0.125, GOOD, 1),
    (1, 1, 128, 96, 0.125, GOOD, 2),
    (1, 1, 128, 32, 0.125, GOOD, 2),
    (1, 1, 128, 64, 0.0, GOOD, 1),
    (1, 1, 128, 64, -1.0, GOOD, 1),
    (1, 1, 128, 64, float("nan"), GOOD, 1),
    (1, 1, 128, 64, float("inf"), GOOD, 1),
    (1, 1, 128, 64, 0.125, 0, 1),
    (1, 1, 128, 64, 0.125, GOOD + 8, 1),
    (4096, 4096, 4096, 64, 0.125, GOOD, 1),
])
def test_fwd_rejects_bad_arguments(lib, B, H, N, d, scale, ptr, want):
    rc = lib.fattn_fwd(ptr, GOOD, GOOD, GOOD, GOOD, B, H, N, d, 0, scale, None)
    assert rc == want


def test_bwd_rejects_bad_arguments(lib):
    need = lib.fattn_bwd_workspace_bytes(1, 1, 128, 64)
    args = [GOOD] * 10
    assert lib.fattn_bwd(*args[:9], GOOD, need - 1, 1, 1, 128, 64, 0, 0.125, None) == 1
    assert lib.fattn_bwd(*args[:9], GOOD + 16, need, 1, 1, 128, 64, 0, 0.125, None) == 1
    assert lib.fattn_bwd(*args[:9], GOOD, need, 1, 1, 128, 80, 0, 0.125, None) == 2
    assert lib.fattn_bwd(*args[:9], GOOD, need, 1, 1, 128, 64, 0, 0.0, None) == 1
    bad = list(args[:9])
    bad[4] = 0
    assert lib.fattn_bwd(*bad, GOOD, need, 1, 1, 128, 64, 0, 0.125, None) == 1
    assert lib.fattn_bwd_preprocess(GOOD, GOOD, GOOD, GOOD + 4, 1, 1, 128, 64, None) == 1


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "missing" / "libfattn.so"))
