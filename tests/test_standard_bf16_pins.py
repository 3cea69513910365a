"""Pins of the bf16 standard-attention baseline (oracle/standard_bf16.py) against facts that do
not come from it:

* ``round_bf16`` against PyTorch's own float32 -> bfloat16 conversion (a library routine,
  round-to-nearest-even) on random values, exact ties and special values, and against ties
  worked out by hand;
* with the rounding switched off, the baseline is exactly the plain definition of attention
  and its gradients (``oracle.attention``, itself pinned in test_oracle_pins.py): a dropped
  term, a transposed operand or a wrong scale in the baseline's formulas fails here;
* with the rounding on, every stored matrix is a bf16 value, and the error against the exact
  result has the size that one bf16 rounding per step predicts: not zero, and far below 1e-1.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.standard_bf16 import round_bf16, standard_attention


def _rand(n, d, seed, sigma=1.0):
    return np.random.default_rng(seed).standard_normal((n, d)) * sigma


def _torch_bf16(x32):
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),       # subnormal fp32
        (rng.standard_normal(2000) * 1e38).astype(np.float32),        # near the fp32 maximum
        np.array([3.39e38, -3.39e38], dtype=np.float32),                # round to +-inf in bf16
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0], dtype=np.float32),
    ])
    # exact ties: the dropped low half is exactly 0x8000, for even and odd kept halves
    hi = (rng.integers(0x0080, 0x7F00, 4000, dtype=np.uint32) << 16)
    ties = (hi | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    got = round_bf16(x)
    ref = _torch_bf16(x)
    assert np.array_equal(got, ref)
    assert np.isnan(round_bf16(np.array([np.nan]))).all()


def test_round_bf16_hand_ties():
    # bf16 keeps 8 significant bits: neighbours of 1 are 1 - 2^-8 and 1 + 2^-7
    assert round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0                    # tie -> even (1)
    assert round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6      # tie -> even
    assert round_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -20]))[0] == 1 + 2.0 ** -7
    assert round_bf16(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0
    assert round_bf16(np.array([3.0]))[0] == 3.0


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 9), (True, 5)])
def test_unrounded_baseline_is_the_definition(causal, kv_len):
    n, d, scale = 13, 8, 0.35
    q, k, v, do = (_rand(n, d, s) for s in (91, 92, 93, 94))
    std = standard_attention(q, k, v, do, scale, causal, kv_len, rounding=False)
    ref = oracle.attention_backward(q, k, v, do, scale, causal, kv_len)
    for name in ("O", "dQ", "dK", "dV"):
        assert np.max(np.abs(std[name] - ref[name])) < 1e-12, name


@pytest.mark.parametrize("causal", [False, True])
def test_rounded_baseline_error_size(causal):
    n, d = 256, 64
    scale = 1.0 / d ** 0.5
    q, k, v, do = (round_bf16(_rand(n, d, s)) for s in (95, 96, 97, 98))
    std = standard_attention(q, k, v, do, scale, causal)
    ref = oracle.attention_backward(q, k, v, do, scale, causal)
    for name in ("S", "P", "O", "dP", "dS", "dQ", "dK", "dV"):
        x = std[name]
        fin = np.isfinite(x)
        assert np.array_equal(round_bf16(x[fin]), x[fin]), name
    for name in ("O", "dQ", "dK", "dV"):
        rel = np.linalg.norm(std[name] - ref[name]) / np.linalg.norm(ref[name])
        assert 1e-4 < rel < 5e-2, (name, rel)
