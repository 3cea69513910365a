"""Host pipeline planning (CPU): the chunks of HostAttention cover every (batch, head) exactly
once, each chunk is one contiguous slice of a [B, H, N, d] tensor, and the count is near the
target."""

import itertools

import pytest

from exact_io_aware_fwd_gb300.pipeline import _chunks, _seq_chunks


@pytest.mark.parametrize("B,H,target", [(1, 32, 16), (1, 32, 8), (16, 16, 16), (64, 16, 16),
                                        (8, 12, 16), (3, 5, 16), (1, 1, 16), (20, 3, 16)])
def test_chunks_partition(B, H, target):
    plan = list(_chunks(B, H, target=target))
    seen = set()
    for b0, b1, h0, h1 in plan:
        assert 0 <= b0 < b1 <= B and 0 <= h0 < h1 <= H
        # contiguous in [B, H, ...]: whole heads of several batches, or a head range of one batch
        assert (h0 == 0 and h1 == H) or b1 == b0 + 1
        for bh in itertools.product(range(b0, b1), range(h0, h1)):
            assert bh not in seen
            seen.add(bh)
    assert len(seen) == B * H
    assert len(plan) <= max(target, B) + H


def test_heads_per_chunk_override():
    plan = list(_chunks(2, 6, heads_per_chunk=4))
    assert plan == [(0, 1, 0, 4), (0, 1, 4, 6), (1, 2, 0, 4), (1, 2, 4, 6)]


@pytest.mark.parametrize("lengths,target", [([512, 4096, 1000, 2000, 3000, 700, 4000, 512] * 2, 16),
                                            ([100] * 40, 16), ([0, 0, 5], 16), ([7], 16),
                                            ([3000, 1, 1, 1, 1, 1], 4), ([5, 0, 9, 0], 2)])
def test_seq_chunks_partition(lengths, target):
    """Runs of whole sequences: contiguous, in order, covering every sequence once, at most
    `target` of them."""
    runs = _seq_chunks(lengths, target=target)
    assert runs[0][0] == 0 and runs[-1][1] == len(lengths)
    assert all(b0 < b1 for b0, b1 in runs)
    assert all(a[1] == b[0] for a, b in zip(runs, runs[1:]))
    assert len(runs) <= target


def test_seq_chunks_balance():
    """Equal sequences split into equal runs; one dominant sequence gets a run of its own."""
    assert _seq_chunks([100] * 16, target=4) == [(0, 4), (4, 8), (8, 12), (12, 16)]
    runs = _seq_chunks([10, 10, 5000, 10, 10], target=3)
    assert any(b1 - b0 == 1 and b0 == 2 for b0, b1 in runs) or (2, 3) in runs
