"""The FLOP counts the bench reports: the nominal convention (4 N^2 d forward, 10 N^2 d backward
per head, halved when causal) and, for key-padded workloads, the count of the (query, key) pairs
that are actually kept, checked against brute-force enumeration of the visible pairs."""

import dataclasses

import pytest
import torch

from exact_io_aware_fwd_gb300.workloads import BY_NAME


def _pairs(N, lens, causal):
    return sum(1 for L in lens for i in range(N) for j in range(N) if j < L and (not causal or j <= i))


@pytest.mark.parametrize("causal", [False, True])
def test_effective_flops_count_visible_pairs(causal):
    w = dataclasses.replace(BY_NAME["ragged-8x12x2000x128"], B=3, H=2, N=50, d=4,
                            kv_len_range=(5, 50), causal=causal)
    lens = torch.tensor([7, 50, 23, 0][:3], dtype=torch.int32)
    f, b = w.flops_effective(lens)
    p = _pairs(50, lens.tolist(), causal) * w.H * w.d
    assert (f, b) == (4.0 * p, 10.0 * p)


def test_effective_equals_nominal_without_padding():
    w = BY_NAME["long-causal-1x32x16384x128"]
    assert w.flops_effective(None) == w.flops()
    full = dataclasses.replace(BY_NAME["ragged-8x12x2000x128"], B=2, H=1, N=64, d=4, causal=False)
    assert full.flops_effective(torch.tensor([64, 64])) == full.flops()
