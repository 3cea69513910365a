"""CPU checks of the C-ABI library: it builds, loads, exports every declared entry point, and
rejects bad arguments synchronously (no kernel is launched by any call here)."""

import ctypes
import os
import re

import pytest

import exact_io_aware_fwd_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def test_header_and_binding_agree():
    assert _declared() == sorted(fa.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(6):
        assert fa.fa_status_string(code)
    assert fa.fa_status_string(4) == "device pipeline wait timed out"


def test_workspace_size(lib):
    # dq accumulator (N padded to 128 rows) + two padded per-row float arrays, 256-byte aligned
    assert fa.fa_bwd_workspace_size(1, 1, 128, 64) == 128 * 64 * 4 + 2 * 512
    n = fa.fa_bwd_workspace_size(2, 3, 2000, 128)
    npad = 2048
    assert n == 6 * npad * 128 * 4 + 2 * ((6 * npad * 4 + 255) // 256 * 256)
    assert fa.fa_bwd_workspace_size(1, 1, 128, 96) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 128, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 0, 64) == 0


def test_invalid_arguments_are_rejected_before_launch(lib):
    p = ctypes.c_void_p(0x10000)  # aligned fake pointer, never dereferenced on these paths
    null = ctypes.c_void_p(0)
    # unsupported head dimension
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 128, 96, 0, -1.0, null, null) == fa.FA_ERR_UNSUPPORTED
    # non-positive sizes
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 0, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd(p, p, p, p, p, 0, 1, 8, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    # null and misaligned pointers
    assert lib.fa_fwd(null, p, p, p, p, 1, 1, 8, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    mis = ctypes.c_void_p(0x10008)
    assert lib.fa_fwd(p, mis, p, p, p, 1, 1, 8, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    # non-finite scale
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 8, 64, 0, float("nan"), null, null) == fa.FA_ERR_INVALID_ARG
    # missing / short workspace
    args = [p] * 9 + [1, 1, 8, 64, 0, -1.0, null]
    assert lib.fa_bwd(*args, null, 1 << 20, null) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(*args, p, 16, null) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_dq_convert(p, 1, 1, 8, 64, -1.0, null, 0, null) == fa.FA_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_library(str(tmp_path / "missing.so"))
