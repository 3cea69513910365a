"""Standard (materialising) attention in bf16: the baseline whose own error sets the yardstick of
the pages' numerical contract.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it.

The contract (page "FlashAttention：不减少一次注意力计算，为什么反而更快", section
"数值精确、低精度与可复现性"; the same criterion, a factor of about 2, on page "FlashAttention 入门：
从 FA1 到 FA4 的 IO 感知注意力", closing list of proposed checks, item 2): a blocked kernel in low
precision is correct when its largest error against an exact reference stays within a small
multiple of the error that the standard implementation, run in the same low precision, makes
against that reference.

What the standard implementation is (first page, section "整体框架：不落盘的完整 attention",
stage table, column of standard attention's HBM objects): S = QK^T / sqrt(d) is written out in
full, read back by the mask + softmax step which writes P in full, and O = P V; the backward
keeps P and reads it again.  Run in bf16, every one of those stored matrices is a bf16 tensor.
The reading taken here (the pages do not spell out the precision of each step): each product
or elementwise step computes in fp32 from bf16 operands and stores its result rounded to bf16,
round-to-nearest-even, as an eager bf16 implementation does:

  S  = bf16(scale * Q K^T)            masked entries -inf
  P  = bf16(softmax(S))               row softmax of the stored S
  O  = bf16(P V)
  dV = bf16(P^T dO)
  dP = bf16(dO V^T)
  dS = bf16(P o (dP - rowsum(P o dP)))  softmax backward from the stored P and dP
  dQ = bf16(scale * dS K),  dK = bf16(scale * dS^T Q)

The fp32 accumulation error inside each product is far below one bf16 rounding and is not
modelled: products and sums are taken in float64, then rounded to fp32 and from fp32 to bf16
(the fp32 step is the accumulator's own precision).  ``rounding=False`` skips every rounding and
returns the exact attention of ``oracle.attention`` (a test pins that identity).
"""

from __future__ import annotations

import numpy as np

from .attention import _f64, masked_scores

__all__ = ["round_bf16", "standard_attention"]


def round_bf16(x):
    """Round to bfloat16 (8 significant bits), round-to-nearest-even, returned as float64.

    The value is first rounded to fp32 (numpy's conversion, nearest-even), then the fp32 bit
    pattern is rounded to its upper 16 bits: add 0x7FFF plus the lowest kept bit and clear the
    low half.  Infinities pass through; a NaN stays a NaN."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rounded = ((bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    out = rounded.view(np.float32).astype(np.float64)
    out[nan] = np.nan
    return out


def _softmax_rows(s):
    """Row softmax of a score matrix with -inf for masked entries; all-masked rows give 0."""
    m = s.max(axis=1)
    p = np.zeros_like(s)
    live = np.isfinite(m)
    if live.any():
        e = np.exp(s[live] - m[live][:, None])
        p[live] = e / e.sum(axis=1)[:, None]
    return p


def standard_attention(q, k, v, do, scale, causal=False, kv_len=None, rounding=True):
    """Forward and backward of standard attention on one [N, d] slice, every stored matrix
    rounded to bf16 when ``rounding`` is true.  Returns a dict with O, dQ, dK, dV (and S, P,
    dP, dS, the stored intermediates); ``do`` may be None for the forward alone."""
    r = round_bf16 if rounding else (lambda a: a)
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = r(masked_scores(q, k, scale, causal, kv_len))
    p = r(_softmax_rows(s))
    out = {"S": s, "P": p, "O": r(p @ v)}
    if do is None:
        return out
    do = _f64(do)
    dv = r(p.T @ do)
    dp = r(do @ v.T)
    ds = r(p * (dp - (p * dp).sum(axis=1)[:, None]))
    out.update(dP=dp, dS=ds, dV=dv, dQ=r(float(scale) * (ds @ k)), dK=r(float(scale) * (ds.T @ q)))
    return out
