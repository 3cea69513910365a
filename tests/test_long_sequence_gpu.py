"""GPU parity at a sequence length far past the benchmark's (N = 131,072, 8x the long causal
workload): the oracle cannot form the N x N matrices, so it checks what it can compute exactly
one piece at a time — O, LSE and dQ of sampled query rows (each needs only its own row of
scores), and, under the causal mask, dK and dV of the last key tile (only the last 128 query
rows reach those keys)."""

import numpy as np
import pytest
import torch

from exact_io_aware_fwd_gb300.workloads import make_inputs
from oracle.attention import key_gradients, row_statistics

from parity import compare_grad, compare_slice, f64, run_gpu

pytestmark = pytest.mark.gpu

N = 131072
ROWS = [0, 1, 127, 128, 4095, 65535, 65536, 98304 + 77, N - 129, N - 128, N - 1]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import exact_io_aware_fwd_gb300 as fa

    fa.build()
    fa.load_library()


@pytest.mark.parametrize("causal", [True, False])
def test_long_sequence_rows_and_last_key_tile(causal):
    d = 128
    q, k, v, do, _ = make_inputs(1, 1, N, d, seed=131)
    out = run_gpu(q, k, v, do, causal, None, None, with_bwd=True)
    scale = 1.0 / d ** 0.5
    qs, ks, vs, dos = (f64(x[0, 0]) for x in (q, k, v, do))
    ref = row_statistics(qs, ks, vs, dos, scale, causal=causal, rows=ROWS)
    got = {name: f64(out[name][0, 0])[ROWS] for name in ("O", "LSE", "dQ")}
    compare_slice(got, ref, f"N={N} causal={causal} rows", with_bwd=False)
    compare_grad(got["dQ"], ref["dQ"], f"N={N} causal={causal} dQ rows")
    if causal:
        last = np.arange(N - 128, N)
        st = row_statistics(qs, ks, vs, dos, scale, causal=True, rows=last)
        kg = key_gradients(qs, ks, vs, dos, scale, st["LSE"], st["D"], causal=True, cols=last,
                           rows=last)
        for name in ("dK", "dV"):
            compare_grad(f64(out[name][0, 0])[last], kg[name], f"N={N} last key tile {name}")
    assert torch.all(torch.isfinite(out["dK"])) and torch.all(torch.isfinite(out["dV"]))
