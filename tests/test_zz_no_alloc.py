"""The allocation-free backward entry point (fa_bwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory (for instance code running inside a host callback or
an allocator hook, or a plugin whose host framework owns every allocation), so fa_bwd_noalloc
takes its workspace from a static device array inside the library.  This test checks that it
gives the same dQ, dK, dV as fa_bwd with a caller-provided workspace, on two calls in a row (the
second call finds the first call's data still in the array), and that sizes beyond the array are
refused before anything runs.  The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_fwd_gb300 as fa
from exact_io_aware_fwd_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

TOL_GRAD_REL = 2e-2  # the gradient tolerance of the parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


@pytest.mark.parametrize("B,H,N,d,causal,kvr", [(2, 3, 700, 128, True, None),
                                                 (2, 2, 517, 64, False, (300, 517))])
def test_noalloc_matches_fa_bwd_twice(B, H, N, d, causal, kvr):
    fa.build()
    lib = fa.load_library()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q, k, v, do, kv = make_inputs(B, H, N, d, seed=17 + N, kv_len_range=kvr)
    q, k, v, do = (t.to(dev) for t in (q, k, v, do))
    kvd = kv.to(dev) if kv is not None else None
    o, lse = fa.fa_fwd(q, k, v, causal=causal, kv_lens=kvd)
    ref = fa.fa_bwd(q, k, v, o, do, lse, causal=causal, kv_lens=kvd)
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk),
                                _p(dv), B, H, N, d, int(causal), -1.0, _p(kvd), stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        assert lib.fa_get_error(stream) == fa.FA_OK
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            assert torch.isfinite(got).all(), (call, name)
            assert _rel(got, want) <= TOL_GRAD_REL, (call, name, _rel(got, want))


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
