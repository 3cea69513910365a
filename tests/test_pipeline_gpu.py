"""GPU: the host pipelines (chunks of whole key/value-head groups or whole sequences, copies
overlapped with compute) give the device path's results for grouped-query and packed
variable-length batches.  Every chunk computes exactly what the whole-batch call computes for
its heads or sequences, so O, LSE, dK and dV match bit for bit, and dQ too with the
deterministic backward (with atomics only the summation order of dQ differs)."""

import pytest
import torch

from exact_io_aware_fwd_gb300 import binding as fa
from exact_io_aware_fwd_gb300.pipeline import HostAttention, VarlenHostAttention
from exact_io_aware_fwd_gb300.workloads import make_gqa_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import exact_io_aware_fwd_gb300 as pkg

    pkg.build()
    pkg.load_library()


def _compare(out, ref, det):
    for name in ("O", "LSE", "dK", "dV"):
        assert torch.equal(out[name], ref[name].cpu()), name
    if det:
        assert torch.equal(out["dQ"], ref["dQ"].cpu())
    else:
        a, b = out["dQ"].double(), ref["dQ"].cpu().double()
        assert torch.linalg.norm(a - b) / torch.linalg.norm(b) < 1e-2


def _gqa_reference(q, k, v, do, causal, det):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.fa_bwd_gqa(qd, kd, vd, o, dod, lse, causal=causal, deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_get_error() == fa.FA_OK
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}


def _varlen_reference(q, k, v, do, cu, max_len, causal, det):
    qd, kd, vd, dod, cud = (t.to(DEV) for t in (q, k, v, do, cu))
    o, lse = fa.fa_fwd_varlen(qd, kd, vd, cud, max_len, causal=causal)
    dq, dk, dv = fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, cud, max_len, causal=causal,
                                  deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_get_error() == fa.FA_OK
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}


@pytest.mark.parametrize("d,causal,det", [(128, True, True), (64, False, False), (128, False, False)])
def test_gqa_pipeline_matches_device_path(d, causal, det):
    B, H, Hkv, N = 2, 8, 2, 300
    q, k, v, do = make_gqa_inputs(B, H, Hkv, N, d, seed=41)
    ref = _gqa_reference(q, k, v, do, causal, det)
    ha = HostAttention(B, H, N, d, Hkv=Hkv, heads_per_chunk=4)  # one key/value head per chunk
    assert len(ha.plan) == B * Hkv
    out = ha.run(*(t.pin_memory() for t in (q, k, v, do)), causal=causal, deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_get_error() == fa.FA_OK
    _compare(out, ref, det)


LENGTHS = [100, 300, 0, 517, 64, 1000, 1, 256]


@pytest.mark.parametrize("d,causal,det,Hkv", [(128, True, True, 4), (64, False, False, 2),
                                              (128, False, True, 1)])
def test_varlen_pipeline_matches_device_path(d, causal, det, Hkv):
    H = 4
    q, k, v, do, cu = make_varlen_inputs(LENGTHS, H, Hkv, d, seed=43)
    ref = _varlen_reference(q, k, v, do, cu, max(LENGTHS), causal, det)
    ha = VarlenHostAttention(cu, H, d, Hkv=Hkv, chunks=4)
    assert len(ha.plan) > 1
    out = ha.run(*(t.pin_memory() for t in (q, k, v, do)), causal=causal, deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_get_error() == fa.FA_OK
    _compare(out, ref, det)


def test_varlen_pipeline_graph_replays():
    """graph=True: the captured run, and a replay after new values are written into the same
    pinned buffers, give the device path's results for the values then in the buffers."""
    H, Hkv, d = 4, 2, 128
    ha = VarlenHostAttention(torch.tensor([0, 100, 400, 400, 917, 981, 1981]), H, d, Hkv=Hkv,
                             chunks=3)
    lengths = [100, 300, 0, 517, 64, 1000]
    bufs = None
    for seed in (51, 52):
        q, k, v, do, cu = make_varlen_inputs(lengths, H, Hkv, d, seed=seed)
        if bufs is None:
            bufs = [t.pin_memory() for t in (q, k, v, do)]
        else:
            for dst, src in zip(bufs, (q, k, v, do)):
                dst.copy_(src)
        out = ha.run(*bufs, causal=True, deterministic=True, graph=True)
        torch.cuda.synchronize()
        got = {n: t.clone() for n, t in out.items()}
        _compare(got, _varlen_reference(q, k, v, do, cu, max(lengths), True, True), True)
