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
    # dq accumulator (N padded to 128 rows) + two padded per-row float arrays + a 16-byte record
    # per 128-row tile, each part 256-byte aligned
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert fa.fa_bwd_workspace_size(1, 1, 128, 64) == 128 * 64 * 4 + 2 * 512 + 256
    n = fa.fa_bwd_workspace_size(2, 3, 2000, 128)
    npad = 2048
    assert n == 6 * npad * 128 * 4 + 2 * up(6 * npad * 4) + up(6 * (npad // 128) * 16)
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
    assert lib.fa_bwd_preprocess(p, p, p, 1, 1, 8, 64, null, 0, null) == fa.FA_ERR_WORKSPACE
    # fa_bwd checks every 16-byte operand pointer (Q, K, V, O, dO, dQ, dK, dV; LSE needs only
    # 4 bytes) before its first launch, and before looking for a device
    for bad in (0, 1, 2, 3, 4, 6, 7, 8):
        bargs = [p] * 9
        bargs[bad] = mis
        rc = lib.fa_bwd(*bargs, 1, 1, 8, 64, 0, -1.0, null, p, 1 << 20, null)
        assert rc == fa.FA_ERR_INVALID_ARG, (bad, rc)


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_library(str(tmp_path / "missing.so"))


def test_invalid_arguments_of_the_extensions(lib):
    """Grouped-query, variable-length and block-sparse entry points reject bad arguments before
    touching the device (this machine may have none)."""
    p = ctypes.c_void_p(0x10000)
    null = ctypes.c_void_p(0)
    mis = ctypes.c_void_p(0x10004)
    # grouped-query: Hkv must divide H
    assert lib.fa_fwd_gqa(p, p, p, p, p, 1, 6, 4, 128, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_gqa(p, p, p, p, p, 1, 6, 0, 128, 64, 0, -1.0, null, null) == fa.FA_ERR_INVALID_ARG
    bargs = [p] * 9 + [1, 6, 4, 128, 64, 0, -1.0, null, 0, p, 1 << 20, null]
    assert lib.fa_bwd_gqa(*bargs) == fa.FA_ERR_INVALID_ARG
    # variable-length: offsets required, sizes checked, an empty batch is a no-op
    assert lib.fa_fwd_varlen(p, p, p, p, p, null, 2, 128, 256, 4, 4, 64, 0, -1.0, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_varlen(p, p, p, p, p, p, 2, 128, -1, 4, 4, 64, 0, -1.0, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_varlen(p, p, p, p, p, p, 2, 0, 256, 4, 4, 64, 0, -1.0, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_varlen(p, p, p, p, p, p, 2, 128, 256, 4, 3, 64, 0, -1.0, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_varlen(null, null, null, null, null, p, 2, 128, 0, 4, 4, 64, 0, -1.0, null) == fa.FA_OK
    assert lib.fa_bwd_varlen_workspace_size(0, 256, 4, 64) == 0
    assert lib.fa_bwd_varlen_workspace_size(2, 256, 4, 96) == 0
    # ceil(256 / 128) + 2 = 4 tiles of 128 rows per head: dQ fp32 + two row statistics
    assert lib.fa_bwd_varlen_workspace_size(2, 256, 4, 64) >= 4 * 4 * 128 * (64 + 2) * 4
    vargs = [p] * 9 + [p, 2, 128, 256, 4, 4, 64, 0, -1.0, 0]
    assert lib.fa_bwd_varlen(*vargs, null, 1 << 20, null) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_varlen(*vargs, p, 16, null) == fa.FA_ERR_WORKSPACE
    # block-sparse: index size, build arguments, mask heads 1 or H, aligned index
    assert lib.fa_block_index_size(0, 1) == 0 and lib.fa_block_index_size(1000, 0) == 0
    t = (1000 + 127) // 128
    tb = (t + 1) // 2
    assert lib.fa_block_index_size(1000, 2) == 2 * 4 * (2 * t * t + 3 * t + tb * (t + 1))
    assert lib.fa_block_index_build(null, 1000, 1, p, 1 << 20, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_block_index_build(p, 1000, 1, mis, 1 << 20, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_block_index_build(p, 1000, 1, p, 16, null) == fa.FA_ERR_WORKSPACE
    assert lib.fa_fwd_block_sparse(p, p, p, p, p, 1, 4, 1000, 64, 0, -1.0, null, p, 3, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_block_sparse(p, p, p, p, p, 1, 4, 1000, 64, 0, -1.0, null, mis, 1, null) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_block_sparse(p, p, p, p, p, 1, 4, 1000, 64, 0, -1.0, null, null, 1, null) == fa.FA_ERR_INVALID_ARG
    sargs = [p] * 9 + [1, 4, 1000, 64, 0, -1.0, null, p, 2, 0]
    assert lib.fa_bwd_block_sparse(*sargs, p, 1 << 20, null) == fa.FA_ERR_INVALID_ARG
