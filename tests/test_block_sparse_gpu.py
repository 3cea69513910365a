"""Block-sparse attention (fa_block_index_build, fa_fwd_block_sparse, fa_bwd_block_sparse) against
the fp64 oracle with the same block mask, on random masks, masks with empty rows and columns,
per-head masks, the causal and key-length masks on top, and the butterfly workload at full size."""

from __future__ import annotations

import pytest
import torch

from exact_io_aware_fwd_gb300.workloads import (SPARSE_WORKLOADS, make_inputs, random_block_mask,
                                                 sample_slices, workload_block_mask,
                                                 workload_inputs)
from parity import check_case, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import exact_io_aware_fwd_gb300 as fa

    fa.build()
    fa.load_library()


CASES = [
    # B, H, N, d, causal, kv range, density, per-head masks
    (1, 2, 640, 128, False, None, 0.5, False),
    (1, 2, 640, 64, True, None, 0.5, False),
    (2, 2, 517, 128, True, (300, 517), 0.6, True),
    (2, 3, 389, 64, False, (1, 389), 0.4, True),
    (1, 1, 1100, 128, False, None, 0.25, False),
    (1, 2, 1100, 64, True, None, 0.3, True),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{'c' if c[4] else ''}s{c[6]}")
def test_random_masks(case, deterministic):
    B, H, N, d, causal, kvr, dens, per_head = case
    T = (N + 127) // 128
    q, k, v, do, kv = make_inputs(B, H, N, d, seed=300 + N + d, kv_len_range=kvr)
    mask = random_block_mask(T, dens, seed=N + d, heads=H if per_head else 1)
    check_case(q, k, v, do, causal, None, kv, label=str(case), deterministic=deterministic,
               block_mask=mask)


@pytest.mark.parametrize("d", [64, 128])
def test_empty_rows_and_columns(d):
    """A query tile with no kept tile gets O = 0, LSE = -inf, dQ = 0; a key tile no query tile
    keeps gets dK = dV = 0."""
    N = 700
    T = (N + 127) // 128
    q, k, v, do, _ = make_inputs(1, 2, N, d, seed=17 + d)
    mask = torch.ones((T, T), dtype=torch.uint8)
    mask[2, :] = 0  # query rows 256..383 keep nothing
    mask[:, 4] = 0  # keys 512..639 are dropped everywhere
    out, _ = check_case(q, k, v, do, False, None, None, label=f"empty d={d}", block_mask=mask)
    assert torch.count_nonzero(out["O"][:, :, 256:384]) == 0
    assert torch.all(torch.isinf(out["LSE"][:, :, 256:384]))
    assert torch.count_nonzero(out["dQ"][:, :, 256:384]) == 0
    assert torch.count_nonzero(out["dK"][:, :, 512:640]) == 0
    assert torch.count_nonzero(out["dV"][:, :, 512:640]) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_all_kept_mask_matches_dense(causal):
    """Keeping every tile visits the same tiles in the same order as the dense forward (bit-equal
    O and LSE); the backward visits the query tiles in another order (equal within rounding)."""
    q, k, v, do, _ = make_inputs(2, 2, 900, 128, seed=23)
    T = (900 + 127) // 128
    a = run_gpu(q, k, v, do, causal, None, None, block_mask=torch.ones((T, T), dtype=torch.uint8))
    b = run_gpu(q, k, v, do, causal, None, None)
    assert torch.equal(a["O"], b["O"]) and torch.equal(a["LSE"], b["LSE"])
    for name in ("dQ", "dK", "dV"):
        rel = torch.linalg.norm(a[name].double() - b[name].double()) / torch.linalg.norm(b[name].double())
        assert rel < 1e-2, (name, float(rel))


def test_deterministic_block_sparse_is_bitwise_repeatable():
    q, k, v, do, _ = make_inputs(1, 4, 2000, 128, seed=29)
    mask = random_block_mask(16, 0.5, seed=31)
    a = run_gpu(q, k, v, do, True, None, None, deterministic=True, block_mask=mask)
    b = run_gpu(q, k, v, do, True, None, None, deterministic=True, block_mask=mask)
    for name in ("O", "LSE", "dQ", "dK", "dV"):
        assert torch.equal(a[name], b[name]), name


def test_index_lists():
    """The index holds, per query block / query tile / key tile, the sorted kept tiles."""
    import exact_io_aware_fwd_gb300 as fa

    N, T = 1000, 8
    mask = random_block_mask(T, 0.4, seed=37)
    idx = fa.fa_block_index_build(mask.cuda(), N).tensor.cpu()
    Tb = (T + 1) // 2
    fcnt, fidx = idx[:Tb], idx[Tb:Tb + Tb * T].view(Tb, T)
    o = Tb + Tb * T
    rcnt, ridx = idx[o:o + T], idx[o + T:o + T + T * T].view(T, T)
    o += T + T * T
    ccnt, cccnt, cidx = idx[o:o + T], idx[o + T:o + 2 * T], idx[o + 2 * T:o + 2 * T + T * T].view(T, T)
    m = mask.bool()
    for i in range(T):
        keep = torch.nonzero(m[i]).flatten()
        assert int(rcnt[i]) == keep.numel() and torch.equal(ridx[i, :keep.numel()], keep.int())
        col = torch.nonzero(m[:, i]).flatten().flip(0)
        assert int(ccnt[i]) == col.numel() and torch.equal(cidx[i, :col.numel()], col.int())
        assert int(cccnt[i]) == int((col >= i).sum())
    for qb in range(Tb):
        rows = m[2 * qb:2 * qb + 2]
        u0 = rows[0]
        u1 = rows[1] if rows.shape[0] > 1 else torch.zeros_like(u0)
        kts = torch.nonzero(u0 | u1).flatten()
        want = kts * 4 + u0[kts].int() + 2 * u1[kts].int()
        assert int(fcnt[qb]) == kts.numel() and torch.equal(fidx[qb, :kts.numel()], want.int())


@pytest.mark.parametrize("w", SPARSE_WORKLOADS, ids=lambda w: w.name)
def test_workloads_full_size(w):
    q, k, v, do, kv = workload_inputs(w)
    check_case(q, k, v, do, w.causal, w.scale, kv, slices=sample_slices(w), label=w.name,
               block_mask=workload_block_mask(w))
