"""The allocation-free backward entry point (fa_bwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory (for instance code running inside a host callback or
an allocator hook, or a plugin whose host framework owns every allocation), so fa_bwd_noalloc
takes its workspace from a static device array inside the library.  These tests check that it
gives the results of fa_bwd with a caller-provided workspace: dK and dV bit for bit (both are
accumulated in a fixed order), dQ within the gradient tolerance of the parity tests and against
the fp64 oracle; on two calls in a row (the second call finds the first call's data still in the
array), after a call of another shape whose inputs filled the array with NaN, and that sizes
beyond the array are refused before anything runs.  The file is named so that pytest collects it
last.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_fwd_gb300 as fa
from exact_io_aware_fwd_gb300.workloads import make_inputs
from parity import compare_grad, f64, oracle_slice

pytestmark = pytest.mark.gpu

TOL_GRAD_REL = 2e-2  # the gradient tolerance of the parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def _problem(B, H, N, d, causal, kvr, seed, nan_do=False):
    dev = torch.device("cuda:0")
    q, k, v, do, kv = make_inputs(B, H, N, d, seed=seed, kv_len_range=kvr)
    if nan_do:
        do = torch.full_like(do, float("nan"))
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    kvd = kv.to(dev) if kv is not None else None
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, kv_lens=kvd)
    return dict(B=B, H=H, N=N, d=d, causal=causal, q=q, k=k, v=v, do=do, kv=kv, qd=qd, kd=kd,
                vd=vd, dod=dod, kvd=kvd, o=o, lse=lse)


def _noalloc(lib, p):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dq, dk, dv = (torch.full_like(p["qd"], float("nan")) for _ in range(3))
    st = lib.fa_bwd_noalloc(_p(p["qd"]), _p(p["kd"]), _p(p["vd"]), _p(p["o"]), _p(p["dod"]),
                            _p(p["lse"]), _p(dq), _p(dk), _p(dv), p["B"], p["H"], p["N"], p["d"],
                            int(p["causal"]), -1.0, _p(p["kvd"]), stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert lib.fa_get_error(stream) == fa.FA_OK
    return dq, dk, dv


def _check_against_fa_bwd_and_oracle(p, got, label):
    ref = fa.fa_bwd(p["qd"], p["kd"], p["vd"], p["o"], p["dod"], p["lse"], causal=p["causal"],
                    kv_lens=p["kvd"])
    dq, dk, dv = got
    assert torch.equal(dk, ref[1]), f"{label}: dK differs from fa_bwd's"
    assert torch.equal(dv, ref[2]), f"{label}: dV differs from fa_bwd's"
    assert torch.isfinite(dq).all(), label
    assert _rel(dq, ref[0]) <= TOL_GRAD_REL, (label, _rel(dq, ref[0]))
    # dQ against the fp64 oracle, every (b, h) slice
    scale = 1.0 / p["d"] ** 0.5
    for b in range(p["B"]):
        kv_len = int(p["kv"][b]) if p["kv"] is not None else None
        for h in range(p["H"]):
            r = oracle_slice(p["q"][b, h].float().numpy(), p["k"][b, h].float().numpy(),
                             p["v"][b, h].float().numpy(), p["do"][b, h].float().numpy(),
                             p["causal"], scale, kv_len, True)
            compare_grad(f64(dq[b, h]), r["dQ"], f"{label} dQ b={b} h={h}")


@pytest.mark.parametrize("B,H,N,d,causal,kvr", [(2, 3, 700, 128, True, None),
                                                 (2, 2, 517, 64, False, (300, 517))])
def test_noalloc_matches_fa_bwd_twice(B, H, N, d, causal, kvr):
    fa.build()
    lib = fa.load_library()
    p = _problem(B, H, N, d, causal, kvr, seed=17 + N)
    for call in range(2):
        _check_against_fa_bwd_and_oracle(p, _noalloc(lib, p), f"call {call}")


def test_noalloc_ignores_what_a_call_of_another_shape_left():
    """A large d = 128 causal call whose dO is all NaN leaves NaN across the array (statistics,
    dQ partial sums); the next call, d = 64 with key lengths (other offsets of every part of the
    array), must not read any of it."""
    fa.build()
    lib = fa.load_library()
    big = _problem(2, 4, 1900, 128, True, None, seed=5, nan_do=True)
    dq, _, _ = _noalloc(lib, big)
    assert torch.isnan(dq).any()  # the array now holds NaN where the next call's data goes
    small = _problem(3, 2, 333, 64, False, (100, 333), seed=6)
    _check_against_fa_bwd_and_oracle(small, _noalloc(lib, small), "after a NaN call")


def test_noalloc_refuses_sizes_beyond_its_array():
    fa.build()
    lib = fa.load_library()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, H, N, d = 1, 1, 140_000, 128  # workspace ~73 MB > the 64 MiB array
    assert fa.fa_bwd_workspace_size(B, H, N, d) > 64 << 20
    # real buffers of the full size, so no launch could read past them even if one happened
    t = [torch.zeros((B, H, N, d), dtype=torch.bfloat16, device=dev) for _ in range(8)]
    lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
    st = lib.fa_bwd_noalloc(_p(t[0]), _p(t[1]), _p(t[2]), _p(t[3]), _p(t[4]), _p(lse), _p(t[5]),
                            _p(t[6]), _p(t[7]), B, H, N, d, 0, -1.0, None, stream)
    assert st == fa.FA_ERR_WORKSPACE
    assert lib.fa_get_error(stream) == fa.FA_OK
    assert all(bool((x == 0).all()) for x in t[5:])  # outputs untouched: nothing ran
