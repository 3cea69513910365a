"""Seeded synthetic attention workloads.

This module only draws inputs; it holds none of the attention arithmetic, so that the CUDA
library's tests and the fp64 oracle can both consume exactly the same tensors.

Recipe (one generator per workload, ``torch.Generator().manual_seed(seed)`` on the CPU):
  1. Q, K, V, dO are drawn in that order with ``torch.randn(B, H, N, d)`` (float32), multiplied
     by their standard deviation and rounded to bfloat16 (round-to-nearest-even);
  2. if the workload has key padding, ``kv_lens = torch.randint(lo, hi + 1, (B,))`` is drawn
     next from the same generator.
Layout: contiguous [B, H, N, d] bfloat16, the order the attention signature uses.

Grouped-query workloads (Hkv < H) draw K and V with Hkv heads: Q [B, H, N, d], K, V
[B, Hkv, N, d], dO [B, H, N, d], in that order.  Variable-length workloads first draw the B
sequence lengths ``torch.randint(lo, hi + 1, (B,))``, then Q, K, V, dO packed as [total, heads, d]
(sequence b = tokens cu[b] .. cu[b+1]-1, cu the running sum of the lengths).

Block-sparse workloads add a block mask over 128 x 128 tiles (uint8 [T, T], T = ceil(N / 128),
nonzero = kept), shared by every batch and head.  The pages name a fixed butterfly pattern for
the block-sparse extension without drawing it; ``butterfly_block_mask`` takes the support of the
butterfly factors: tile (i, j) is kept when i and j differ in at most one bit, so every row keeps
its diagonal tile and the tiles at distance 2^k in the butterfly sense (1 + log2 T per row when T
is a power of two).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma_qk: float = 1.0
    sigma_vdo: float = 1.0
    kv_len_range: tuple | None = None  # inclusive (lo, hi) of per-batch key lengths
    oracle_slices: int = 0  # (batch, head) slices the oracle checks at full size (0 = all)
    block_mask: str | None = None  # "butterfly": block-sparse over 128 x 128 tiles
    Hkv: int | None = None  # key/value heads (grouped-query attention) when set
    seqlen_range: tuple | None = None  # variable-length: B packed sequences, lengths U{lo..hi}
    notes: str = field(default="", compare=False)

    @property
    def kv_heads(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5

    def flops(self) -> tuple[float, float]:
        """(forward, backward) FLOPs: 4 N^2 d and 10 N^2 d per head, halved when causal.  With a
        block mask N^2 becomes the area of the kept tiles (a causal diagonal tile counts half)."""
        if self.seqlen_range is not None:  # sum of per-sequence N^2 over the packed batch
            lens = draw_lengths(self).double()
            per_head = float((lens * lens).sum()) * self.d
            f, b = 4.0 * per_head * self.H, 10.0 * per_head * self.H
            return (f / 2, b / 2) if self.causal else (f, b)
        if self.block_mask is not None:
            bm = workload_block_mask(self).bool()
            t = bm.shape[0]
            sizes = torch.tensor([min(128, self.N - 128 * i) for i in range(t)], dtype=torch.float64)
            area = sizes[:, None] * sizes[None, :]
            if self.causal:
                area = torch.where(torch.eye(t, dtype=torch.bool), area / 2, area)
                bm = bm & torch.tril(torch.ones(t, t, dtype=torch.bool))
            per_head = float((area * bm).sum()) * self.d
            return 4.0 * per_head * self.B * self.H, 10.0 * per_head * self.B * self.H
        per_head = float(self.N) * self.N * self.d
        f = 4.0 * per_head * self.B * self.H
        b = 10.0 * per_head * self.B * self.H
        if self.causal:
            f, b = f / 2, b / 2
        return f, b

    def flops_effective(self, kv_lens) -> tuple[float, float]:
        """(forward, backward) FLOPs of the (query, key) pairs a key-padded workload actually
        keeps, given its drawn key lengths (workload_inputs' last item): 4 d and 10 d per visible
        pair, N * len_b pairs per head of batch b (causal: the pairs with key <= query among the
        first len_b keys).  The kernels skip the key tiles at or past len_b, so this, not the
        nominal N^2 count, is the work they do.  Without key lengths: flops()."""
        if kv_lens is None or self.kv_len_range is None:
            return self.flops()
        lens = torch.as_tensor(kv_lens).double().clamp(0, self.N)
        n = float(self.N)
        if self.causal:  # sum over queries i of min(i + 1, len_b)
            pairs = lens * (lens + 1) / 2 + (n - lens) * lens
        else:
            pairs = n * lens
        per_head_sum = float(pairs.sum()) * self.d  # summed over the batch
        return 4.0 * per_head_sum * self.H, 10.0 * per_head_sum * self.H


# The five synthetic shapes: a one-head smoke test, the GPT-2-medium attention shape the pages
# time on A100, a causal mid-length case, the long-context causal case the roofline is quoted
# on, and a ragged key-padded stress case with large logits.
WORKLOADS = [
    Workload("smoke-1x1x128x64", 1, 1, 128, 64, False, seed=0),
    Workload("gpt2-medium-64x16x1024x64", 64, 16, 1024, 64, False, seed=1, oracle_slices=4),
    Workload("causal-16x16x4096x128", 16, 16, 4096, 128, True, seed=2, oracle_slices=4),
    Workload("long-causal-1x32x16384x128", 1, 32, 16384, 128, True, seed=3, oracle_slices=2),
    Workload("ragged-8x12x2000x128", 8, 12, 2000, 128, False, seed=4, sigma_qk=3.0,
             kv_len_range=(1000, 2000), oracle_slices=8),
]

# Block-sparse: the long-context shape, non-causal, with the butterfly block mask (8 of 128
# tiles per row, 6.25% of the dense work).
SPARSE_WORKLOADS = [
    Workload("butterfly-1x32x16384x128", 1, 32, 16384, 128, False, seed=5, oracle_slices=2,
             block_mask="butterfly"),
]

# Grouped-query attention on the long-context shape (8 key/value heads for 32 query heads), and a
# packed batch of 16 causal sequences of 512..4096 tokens (N is the longest allowed length).
GQA_WORKLOADS = [
    Workload("gqa-1x32kv8x16384x128", 1, 32, 16384, 128, True, seed=6, oracle_slices=2, Hkv=8),
]
VARLEN_WORKLOADS = [
    Workload("varlen-16x16x512-4096x128", 16, 16, 4096, 128, True, seed=7, oracle_slices=3,
             seqlen_range=(512, 4096)),
]

BY_NAME = {w.name: w for w in WORKLOADS + SPARSE_WORKLOADS + GQA_WORKLOADS + VARLEN_WORKLOADS}
HEADLINE = WORKLOADS[3]


def make_inputs(B, H, N, d, seed, sigma_qk=1.0, sigma_vdo=1.0, kv_len_range=None):
    """Draw (q, k, v, do, kv_lens) on the CPU; kv_lens is None without key padding."""
    g = torch.Generator().manual_seed(int(seed))

    def draw(sigma):
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(torch.bfloat16)

    q = draw(sigma_qk)
    k = draw(sigma_qk)
    v = draw(sigma_vdo)
    do = draw(sigma_vdo)
    kv_lens = None
    if kv_len_range is not None:
        lo, hi = kv_len_range
        kv_lens = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return q, k, v, do, kv_lens


def workload_inputs(w: Workload):
    """(q, k, v, do, extra): extra is kv_lens (dense, may be None) or cu_seqlens (variable-length,
    int32 [B + 1], tensors packed [total, heads, d])."""
    if w.seqlen_range is not None:
        return make_varlen_inputs(draw_lengths(w), w.H, w.kv_heads, w.d, w.seed)
    if w.Hkv is not None:
        return make_gqa_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.seed) + (None,)
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.sigma_qk, w.sigma_vdo, w.kv_len_range)


def make_gqa_inputs(B, H, Hkv, N, d, seed):
    """(q, k, v, do) with q, do [B, H, N, d] and k, v [B, Hkv, N, d], all N(0, 1) in bf16."""
    g = torch.Generator().manual_seed(int(seed))
    shapes = [(B, H, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, H, N, d)]
    return tuple(torch.randn(sh, generator=g).to(torch.bfloat16) for sh in shapes)


def draw_lengths(w: Workload) -> torch.Tensor:
    """The B sequence lengths of a variable-length workload (int32, from its own seed)."""
    lo, hi = w.seqlen_range
    g = torch.Generator().manual_seed(int(w.seed))
    return torch.randint(lo, hi + 1, (w.B,), generator=g).to(torch.int32)


def make_varlen_inputs(lengths, H, Hkv, d, seed):
    """(q, k, v, do, cu_seqlens): sequences of the given lengths packed as [total, heads, d]."""
    lengths = torch.as_tensor(lengths, dtype=torch.int32)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0)
    total = int(cu[-1])
    g = torch.Generator().manual_seed(int(seed) + 1)
    shapes = [(total, H, d), (total, Hkv, d), (total, Hkv, d), (total, H, d)]
    q, k, v, do = (torch.randn(sh, generator=g).to(torch.bfloat16) for sh in shapes)
    return q, k, v, do, cu


def sample_slices(w: Workload, count=None, seed_offset=1000):
    """Seeded choice of (b, h) slices the oracle checks at full size (a separate generator)."""
    count = w.oracle_slices if count is None else count
    total = w.B * w.H
    if count <= 0 or count >= total:
        return [(bh // w.H, bh % w.H) for bh in range(total)]
    g = torch.Generator().manual_seed(w.seed + seed_offset)
    if count == w.B:
        # one head per batch: every drawn key length is covered
        heads = torch.randint(0, w.H, (w.B,), generator=g).tolist()
        return [(b, h) for b, h in enumerate(heads)]
    picks = torch.randperm(total, generator=g)[:count].tolist()
    return [(bh // w.H, bh % w.H) for bh in sorted(picks)]


def butterfly_block_mask(T: int) -> torch.Tensor:
    """uint8 [T, T]: tile (i, j) kept when i XOR j has at most one bit set."""
    i = torch.arange(T)
    x = i[:, None] ^ i[None, :]
    return ((x & (x - 1)) == 0).to(torch.uint8)


def random_block_mask(T: int, density: float, seed: int, heads: int = 1) -> torch.Tensor:
    """uint8 [heads, T, T] (or [T, T] for heads == 1), each tile kept with probability density."""
    g = torch.Generator().manual_seed(int(seed))
    m = (torch.rand((heads, T, T), generator=g) < density).to(torch.uint8)
    return m[0] if heads == 1 else m


def workload_block_mask(w: Workload) -> torch.Tensor | None:
    if w.block_mask is None:
        return None
    if w.block_mask == "butterfly":
        return butterfly_block_mask((w.N + 127) // 128)
    raise ValueError(f"unknown block mask {w.block_mask!r}")

