"""The pages' numerical contract for a low-precision attention kernel: its largest error against
an exact reference stays within about twice the largest error of the standard implementation
run in the same precision (page "FlashAttention：不减少一次注意力计算，为什么反而更快", section
"数值精确、低精度与可复现性").

Exact reference: the fp64 oracle.  Standard implementation: ``oracle.standard_bf16`` (S, P, O
and the backward's dP, dS and gradients stored in bf16).  For O, dQ, dK and dV of each slice the
test computes max |GPU - exact| and max |standard - exact|, prints the ratio, and asserts the
factor 2.  Slices: the smoke shape in full, and seeded (b, h) slices of the GPT-2-medium, causal
4k and key-padded workloads at full size (the 16k shape's N x N matrices are too large for the
materialising baseline).
"""

import numpy as np
import pytest
import torch

from exact_io_aware_fwd_gb300.workloads import BY_NAME, workload_inputs
from oracle.standard_bf16 import standard_attention

from parity import f64, oracle_slice, run_gpu

pytestmark = pytest.mark.gpu
FACTOR = 2.0

CASES = [
    ("smoke-1x1x128x64", [(0, 0)]),
    ("gpt2-medium-64x16x1024x64", [(0, 0), (63, 15)]),
    ("causal-16x16x4096x128", [(5, 9)]),
    ("ragged-8x12x2000x128", [(0, 0), (7, 11)]),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import exact_io_aware_fwd_gb300 as fa

    fa.build()
    fa.load_library()


@pytest.mark.parametrize("name,slices", CASES, ids=[c[0] for c in CASES])
def test_error_within_twice_standard_bf16(name, slices):
    w = BY_NAME[name]
    q, k, v, do, kv = workload_inputs(w)
    out = run_gpu(q, k, v, do, w.causal, None, kv, with_bwd=True)
    torch.cuda.synchronize()
    report = []
    for b, h in slices:
        kv_len = int(kv[b]) if kv is not None else None
        args = [x[b, h].float().numpy() for x in (q, k, v, do)]
        exact = oracle_slice(*args, w.causal, w.scale, kv_len, True)
        std = standard_attention(*args, w.scale, w.causal, kv_len)
        for out_name in ("O", "dQ", "dK", "dV"):
            err_gpu = float(np.max(np.abs(f64(out[out_name][b, h]) - exact[out_name])))
            err_std = float(np.max(np.abs(std[out_name] - exact[out_name])))
            report.append((b, h, out_name, err_gpu, err_std, err_gpu / err_std))
    for b, h, out_name, e_gpu, e_std, ratio in report:
        print(f"{name} b={b} h={h} {out_name}: max err GPU {e_gpu:.3e}, standard bf16 {e_std:.3e}, "
              f"ratio {ratio:.2f}")
    bad = [r for r in report if r[3] > FACTOR * r[4]]
    assert not bad, bad
