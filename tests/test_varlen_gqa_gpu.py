"""Grouped-query attention (fa_fwd_gqa / fa_bwd_gqa) and packed variable-length batches
(fa_fwd_varlen / fa_bwd_varlen) against the fp64 oracle: every query head is checked with its
key/value head, and dK, dV of a shared head against the sum of its group's oracle gradients;
every packed sequence is checked as its own attention problem."""

from __future__ import annotations

import pytest
import torch

from exact_io_aware_fwd_gb300.workloads import (GQA_WORKLOADS, VARLEN_WORKLOADS, make_gqa_inputs,
                                                 make_inputs, make_varlen_inputs, workload_inputs)
from parity import check_heads, f64, run_gpu

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import exact_io_aware_fwd_gb300 as fa

    fa.build()
    fa.load_library()


def run_gqa(q, k, v, do, causal, kv_lens=None, deterministic=False):
    import exact_io_aware_fwd_gb300 as fa

    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    kv = kv_lens.to(DEV) if kv_lens is not None else None
    o, lse = fa.fa_fwd_gqa(qd, kd, vd, causal=causal, kv_lens=kv)
    dq, dk, dv = fa.fa_bwd_gqa(qd, kd, vd, o, dod, lse, causal=causal, kv_lens=kv,
                               deterministic=deterministic)
    assert fa.fa_get_error() == fa.FA_OK
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}


def check_gqa_out(q, k, v, do, out, causal, kv_lens, kv_slices, label):
    H, Hkv, d = q.shape[1], k.shape[1], q.shape[3]
    G = H // Hkv
    for b, hk in kv_slices:
        heads = range(hk * G, hk * G + G)
        got = [{"O": f64(out["O"][b, h]), "LSE": f64(out["LSE"][b, h]), "dQ": f64(out["dQ"][b, h]),
                "dK": f64(out["dK"][b, hk]), "dV": f64(out["dV"][b, hk])} for h in heads]
        kv_len = int(kv_lens[b]) if kv_lens is not None else None
        check_heads([q[b, h] for h in heads], k[b, hk], v[b, hk], [do[b, h] for h in heads], got,
                    causal, 1.0 / d ** 0.5, kv_len, f"{label} b={b} hk={hk}")


GQA_CASES = [
    # B, H, Hkv, N, d, causal, kv range
    (2, 8, 2, 300, 128, True, None),
    (2, 8, 1, 300, 64, False, None),
    (1, 6, 3, 517, 128, False, (200, 517)),
    (2, 4, 2, 640, 64, True, None),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("case", GQA_CASES, ids=lambda c: f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}d{c[4]}{'c' if c[5] else ''}")
def test_gqa_small(case, deterministic):
    B, H, Hkv, N, d, causal, kvr = case
    q, k, v, do = make_gqa_inputs(B, H, Hkv, N, d, seed=400 + N + d)
    kv = None
    if kvr is not None:
        g = torch.Generator().manual_seed(N)
        kv = torch.randint(kvr[0], kvr[1] + 1, (B,), generator=g).to(torch.int32)
    out = run_gqa(q, k, v, do, causal, kv, deterministic)
    check_gqa_out(q, k, v, do, out, causal, kv, [(b, hk) for b in range(B) for hk in range(Hkv)],
                  str(case))


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_with_all_heads_is_plain_attention(causal):
    """Hkv == H visits the same tiles in the same order as fa_fwd / fa_bwd: equal bit for bit
    (dQ through fp32 atomics: equal within rounding)."""
    q, k, v, do, _ = make_inputs(2, 4, 700, 128, seed=41)
    a = run_gqa(q, k, v, do, causal)
    b = run_gpu(q, k, v, do, causal, None, None)
    for name in ("O", "LSE", "dK", "dV"):
        assert torch.equal(a[name], b[name]), name
    rel = torch.linalg.norm(a["dQ"].double() - b["dQ"].double()) / torch.linalg.norm(b["dQ"].double())
    assert rel < 1e-2


def run_varlen(q, k, v, do, cu, max_seqlen, causal, deterministic=False, bufs=None):
    import exact_io_aware_fwd_gb300 as fa

    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    cud = cu.to(DEV)
    bufs = bufs or {}
    o, lse = fa.fa_fwd_varlen(qd, kd, vd, cud, max_seqlen, causal=causal, out=bufs.get("O"),
                              lse=bufs.get("LSE"))
    dq, dk, dv = fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, cud, max_seqlen, causal=causal,
                                  deterministic=deterministic, dq=bufs.get("dQ"),
                                  dk=bufs.get("dK"), dv=bufs.get("dV"))
    assert fa.fa_get_error() == fa.FA_OK
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}


def check_varlen_out(q, k, v, do, cu, out, causal, seqs, label, grad_tol=None):
    H, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    G = H // Hkv
    for b in seqs:
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        for hk in range(Hkv):
            heads = range(hk * G, hk * G + G)
            got = [{"O": f64(out["O"][s0:s1, h]), "LSE": f64(out["LSE"][h, s0:s1]),
                    "dQ": f64(out["dQ"][s0:s1, h]), "dK": f64(out["dK"][s0:s1, hk]),
                    "dV": f64(out["dV"][s0:s1, hk])} for h in heads]
            check_heads([q[s0:s1, h] for h in heads], k[s0:s1, hk], v[s0:s1, hk],
                        [do[s0:s1, h] for h in heads], got, causal, 1.0 / d ** 0.5, None,
                        f"{label} seq={b} hk={hk}", grad_tol)


VARLEN_CASES = [
    # lengths, H, Hkv, d, causal
    ([130, 1, 0, 517, 256], 4, 4, 128, True),
    ([130, 1, 0, 517, 256], 4, 2, 64, False),
    ([300, 700, 129], 2, 1, 128, False),
    ([1000, 37, 383], 4, 4, 64, True),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("case", VARLEN_CASES, ids=lambda c: f"L{len(c[0])}H{c[1]}kv{c[2]}d{c[3]}{'c' if c[4] else ''}")
def test_varlen_small(case, deterministic):
    lengths, H, Hkv, d, causal = case
    q, k, v, do, cu = make_varlen_inputs(lengths, H, Hkv, d, seed=500 + d + len(lengths))
    out = run_varlen(q, k, v, do, cu, max(lengths), causal, deterministic)
    # a one-token sequence has a single key: its gradients are rounding-level (see the edge
    # lengths of the dense tests); the tolerance there is the few-key one
    tol = 5e-2 if min(x for x in lengths if x > 0) < 16 else None
    check_varlen_out(q, k, v, do, cu, out, causal, range(len(lengths)), str(case), tol)


def test_varlen_writes_only_its_rows():
    """Outputs live in larger buffers: rows past `total` keep their canary values."""
    import exact_io_aware_fwd_gb300 as fa

    lengths, H, d = [200, 57, 300], 2, 128
    q, k, v, do, cu = make_varlen_inputs(lengths, H, H, d, seed=61)
    total, extra = sum(lengths), 256
    big = {name: torch.full((total + extra, H, d), 7.0, dtype=torch.bfloat16, device=DEV)
           for name in ("O", "dQ", "dK", "dV")}
    lse_big = torch.full((H, total + extra), 7.0, device=DEV)
    bufs = {name: t[:total] for name, t in big.items()}
    bufs["LSE"] = torch.empty((H, total), device=DEV)
    out = run_varlen(q, k, v, do, cu, max(lengths), True, bufs=bufs)
    for name, t in big.items():
        assert torch.all(t[total:] == 7.0), name
    del lse_big
    check_varlen_out(q, k, v, do, cu, out, True, range(3), "canary")


def test_varlen_deterministic_is_bitwise_repeatable():
    q, k, v, do, cu = make_varlen_inputs([900, 1500, 77, 2048], 4, 2, 128, seed=67)
    a = run_varlen(q, k, v, do, cu, 2048, True, deterministic=True)
    b = run_varlen(q, k, v, do, cu, 2048, True, deterministic=True)
    for name in a:
        assert torch.equal(a[name], b[name]), name


def test_varlen_of_equal_lengths_matches_dense():
    """Equal-length packed sequences are a plain batch: same O, LSE as fa_fwd on [B, H, N, d]."""
    import exact_io_aware_fwd_gb300 as fa

    B, H, N, d = 3, 2, 384, 128
    q, k, v, do, _ = make_inputs(B, H, N, d, seed=71)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()  # noqa: E731
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32)
    out = run_varlen(pack(q), pack(k), pack(v), pack(do), cu, N, True)
    ref = run_gpu(q, k, v, do, True, None, None)
    assert torch.equal(out["O"], pack(ref["O"]))
    assert torch.equal(out["LSE"], ref["LSE"].permute(1, 0, 2).reshape(H, B * N))
    assert torch.equal(out["dK"], pack(ref["dK"])) and torch.equal(out["dV"], pack(ref["dV"]))


def test_varlen_empty_batch():
    import exact_io_aware_fwd_gb300 as fa

    q = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    cu = torch.zeros(3, dtype=torch.int32, device=DEV)
    o, lse = fa.fa_fwd_varlen(q, q, q, cu, 1)
    dq, dk, dv = fa.fa_bwd_varlen(q, q, q, o, q, lse, cu, 1)
    assert fa.fa_get_error() == fa.FA_OK and o.numel() == 0


@pytest.mark.parametrize("w", GQA_WORKLOADS, ids=lambda w: w.name)
def test_gqa_workload_full_size(w):
    q, k, v, do, _ = workload_inputs(w)
    out = run_gqa(q, k, v, do, w.causal)
    check_gqa_out(q, k, v, do, out, w.causal, None, [(0, 3)], w.name)


@pytest.mark.parametrize("w", VARLEN_WORKLOADS, ids=lambda w: w.name)
def test_varlen_workload_full_size(w):
    q, k, v, do, cu = workload_inputs(w)
    out = run_varlen(q, k, v, do, cu, w.N, w.causal)
    # three sequences (the shortest, the longest and the first), every head
    lens = (cu[1:] - cu[:-1]).tolist()
    seqs = sorted({0, lens.index(min(lens)), lens.index(max(lens))})
    check_varlen_out(q[:, :2], k[:, :2], v[:, :2], do[:, :2], cu,
                     {n: (t[:, :2] if n != "LSE" else t[:2]) for n, t in out.items()},
                     w.causal, seqs, w.name)
