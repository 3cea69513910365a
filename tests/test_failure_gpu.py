"""Failure detection without a GPU fault: bounded pipeline waits that run out.

The library's kernels bound every mbarrier wait (sm103.cuh, mbar_wait).  Two forms:
  * a test-only kernel built from tests/csrc/ waits on an mbarrier that nothing arrives on: the
    wait must give up after its limit, record the timeout code (FA_ERR_TIMEOUT = 4) in the status
    word, make the CTA's other role give up through the shared abort flag, and return normally;
  * the library's own kernels run with a wait limit of one microsecond, shorter than the normal
    waits of their pipelines, so that waits run out at whatever point they happen to: every CTA
    must leave through its timeout path (waiting for its own copies and MMAs before it exits),
    the call must report FA_ERR_TIMEOUT, and the next call in the same context, with the normal
    limit, must match the oracle.
"""

import ctypes
import os
import subprocess
import time

import pytest
import torch

import exact_io_aware_fwd_gb300 as fa
from exact_io_aware_fwd_gb300 import build_lib
from exact_io_aware_fwd_gb300.workloads import make_inputs
from parity import check_case

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    fa.load_library()


@pytest.fixture(scope="module")
def selftest_lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("selftest") / "libwait_selftest.so"
    cmd = [build_lib._nvcc(), *build_lib.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-I", build_lib.CSRC, os.path.join(HERE, "csrc", "wait_timeout_selftest.cu"),
           "-o", str(out)]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.wait_timeout_selftest.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong)]
    lib.wait_timeout_selftest.restype = ctypes.c_int
    return lib


def test_dead_wait_times_out_and_context_survives(selftest_lib):
    elapsed = (ctypes.c_ulonglong * 2)()
    t0 = time.time()
    st = selftest_lib.wait_timeout_selftest(50, elapsed)
    wall = time.time() - t0
    assert st == fa.FA_ERR_TIMEOUT, st
    assert wall < 10.0
    # the waiting role gave up after its own 50 ms limit ...
    assert 50e6 <= elapsed[0] < 2e9, elapsed[0]
    # ... and the other role through the abort flag, long before its own 50 s limit
    assert 0 < elapsed[1] < 5e9, elapsed[1]
    # the context is intact: the library still computes correctly afterwards
    q = torch.randn(1, 2, 256, 64, device="cuda").to(torch.bfloat16)
    o, lse = fa.fa_fwd(q, q, q, causal=True)
    assert fa.fa_get_error() == fa.FA_OK
    ref = torch.nn.functional.scaled_dot_product_attention(q.float(), q.float(), q.float(),
                                                           is_causal=True)
    assert torch.max(torch.abs(o.float() - ref)) < 2e-2


@pytest.mark.parametrize("entry,d,causal", [("fwd", 128, True), ("fwd", 64, False),
                                            ("bwd", 128, True), ("bwd", 64, False),
                                            ("bwd_deterministic", 128, True)])
def test_library_kernels_time_out_then_recover(entry, d, causal, monkeypatch):
    B, H, N = 1, 2, 1000
    q, k, v, do, _ = make_inputs(B, H, N, d, seed=41)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal)
    assert fa.fa_get_error() == fa.FA_OK
    monkeypatch.setenv("FA_WAIT_TIMEOUT_US", "1")
    t0 = time.time()
    if entry == "fwd":
        fa.fa_fwd(qd, kd, vd, causal=causal)
    elif entry == "bwd":
        fa.fa_bwd(qd, kd, vd, o, dod, lse, causal=causal)
    else:
        fa.fa_bwd_deterministic(qd, kd, vd, o, dod, lse, causal=causal)
    st = fa.fa_get_error()
    wall = time.time() - t0
    monkeypatch.delenv("FA_WAIT_TIMEOUT_US")
    assert st == fa.FA_ERR_TIMEOUT, fa.fa_status_string(st)
    assert wall < 10.0
    # the same context, the normal limit: every output matches the oracle again
    check_case(q, k, v, do, causal, None, None, label=f"after {entry} timeout",
               deterministic=(entry == "bwd_deterministic"))
