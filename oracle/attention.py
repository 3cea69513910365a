"""fp64 CPU oracle for exact scaled-dot-product attention and its backward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  The library (``exact_io_aware_fwd_gb300``) never
imports it and shares no code with it.

What it computes is the plain definition of attention, which the tiled method reaches exactly up
to rounding order ("Theorem 1": the blocked computation returns softmax(QK^T)V):

* scores      S = scale * Q K^T                 (page "FlashAttention：不减少一次注意力计算，为什么反而更快",
                                                 section 关键设计一, first display equation)
* row softmax P = softmax(S), O = P V           (same equation)
* statistic   LSE = m + log(l), natural log of the scaled scores
                                                (same page, 关键设计二, state table row "FA2 的 L=m+log l")
* backward    dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P o (dP - D),
              dV = P^T dO, dQ = scale * dS K, dK = scale * dS^T Q
                                                (same page, 关键设计三, display equation for D_i and dS_ij)

Masks (both written as score = -inf, i.e. probability exactly 0):
* causal: key j > query i is masked  (page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力",
  section "FlashAttention-1：分块与在线 softmax", paragraph on causal masking: skip blocks j > i);
* key padding: key j >= kv_len is masked (first page, 使用契约 table row "mask/dropout").

* block mask (block-sparse attention): the scores of query i and key j are kept only where
  block_mask[i // block, j // block] is nonzero, every other score is masked.  The extension
  skips the zero blocks and stays exact inside the kept ones (page "FlashAttention 入门：从 FA1
  到 FA4 的 IO 感知注意力", section "FlashAttention-1：分块与在线 softmax", paragraph after the
  causal note; first page, sections "作者团队与论文的系统研究脉络" and "IO 复杂度、内存复杂度与
  exactness 的边界", IO = Theta(Nd + N^2 d^2 s / M) for a fraction s of nonzero blocks).  The
  masks combine: an entry counts only if every mask keeps it.

A row with no unmasked key (reachable with kv_len == 0, or a block mask whose row keeps no
visible block) has O = 0, LSE = -inf and zero gradients; this convention is the oracle's own,
the pages do not define it.

The second forward route, ``tiled_forward``, restates the pages' online-softmax recurrence
(running max m, running sum l, unnormalised output O~, one final divide) in the order the
tutorial page gives it (page "FlashAttention: Fast and Memory-Efficient Exact Attention with
IO-Awareness", section "前向过程").  It exists so that tests can pin the recurrence against the
worked example printed on that page and against the plain definition above.

Everything is float64.  Inputs are converted with ``np.asarray(x, dtype=np.float64)``; callers
pass the bf16-rounded tensors so that both sides see identical inputs.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "masked_scores",
    "row_logsumexp",
    "probabilities",
    "row_statistics",
    "key_gradients",
    "attention_forward",
    "attention_backward",
    "tiled_forward",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _mask(rows, keys, causal, kv_len, block_mask, block):
    """Boolean [len(rows), len(keys)]: True where the score of (row, key) is masked."""
    masked = np.zeros((rows.shape[0], keys.shape[0]), dtype=bool)
    if causal:
        masked |= keys[None, :] > rows[:, None]
    if kv_len is not None:
        masked |= keys[None, :] >= int(kv_len)
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        masked |= ~bm[(rows // block)[:, None], (keys // block)[None, :]]
    return masked


def masked_scores(q, k, scale, causal=False, kv_len=None, rows=None, block_mask=None, block=128):
    """S[rows, :] = scale * Q[rows] K^T with masked entries set to -inf.

    q: [N_q, d], k: [N_k, d].  ``rows`` selects query rows (default: all); the causal mask
    compares the key index with the *absolute* query index, so a row subset gives exactly the
    corresponding rows of the full matrix.  ``block_mask`` ([ceil(N_q / block), ceil(N_k /
    block)], nonzero = kept) masks every entry of a zero block.
    """
    q = _f64(q)
    k = _f64(k)
    n_q, n_k = q.shape[0], k.shape[0]
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    s = float(scale) * (q[rows] @ k.T)
    s[_mask(rows, np.arange(n_k), causal, kv_len, block_mask, block)] = -np.inf
    return s


def row_logsumexp(s):
    """LSE_i = m_i + log(sum_j exp(s_ij - m_i)), m_i = max_j s_ij; -inf for an all-masked row."""
    m = s.max(axis=1)
    lse = np.full(s.shape[0], -np.inf)
    live = np.isfinite(m)
    if live.any():
        ml = m[live]
        lse[live] = ml + np.log(np.exp(s[live] - ml[:, None]).sum(axis=1))
    return lse


def probabilities(s, lse):
    """P_ij = exp(s_ij - LSE_i); exactly 0 for masked entries and for all-masked rows."""
    p = np.zeros_like(s)
    live = np.isfinite(lse)
    if live.any():
        p[live] = np.exp(s[live] - lse[live][:, None])
    return p


def row_statistics(q, k, v, do, scale, causal=False, kv_len=None, rows=None, block_mask=None,
                   block=128):
    """Everything that is local to a set of query rows.

    Returns a dict with, for the selected rows:
      O   [r, d]   softmax(S) V
      LSE [r]      log-sum-exp of the scaled, masked scores
      D   [r]      sum_j P_ij dP_ij   (softmax Jacobian contraction, dP = dO V^T)
      dQ  [r, d]   scale * dS K, dS = P o (dP - D)
    ``do`` may be None, in which case only O and LSE are returned.
    """
    v = _f64(v)
    rows_idx = np.arange(_f64(q).shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    s = masked_scores(q, k, scale, causal, kv_len, rows_idx, block_mask, block)
    lse = row_logsumexp(s)
    p = probabilities(s, lse)
    out = {"O": p @ v, "LSE": lse}
    if do is None:
        return out
    do_r = _f64(do)[rows_idx]
    dp = do_r @ v.T
    d_row = (p * dp).sum(axis=1)
    ds = p * (dp - d_row[:, None])
    out["D"] = d_row
    out["dQ"] = float(scale) * (ds @ _f64(k))
    return out


def key_gradients(q, k, v, do, scale, lse, d_row, causal=False, kv_len=None, cols=None,
                  rows=None, block_mask=None, block=128):
    """dK[cols], dV[cols] as sums over the query rows ``rows`` (default: all rows).

    dV_j = sum_i P_ij dO_i,  dK_j = scale * sum_i dS_ij Q_i,  with P_ij = exp(s_ij - LSE_i) and
    dS_ij = P_ij (dP_ij - D_i), dP_ij = dO_i . V_j.  ``lse`` and ``d_row`` are the statistics of
    the rows summed over (as returned by ``row_statistics`` for the same rows); summing the
    results over a partition of the rows gives the full gradients.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    n_q, n_k = q.shape[0], k.shape[0]
    cols = np.arange(n_k) if cols is None else np.asarray(cols, dtype=np.int64)
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    q = q[rows]
    do = do[rows]
    # scores of the summed query rows against the selected keys, masked like masked_scores
    s = float(scale) * (q @ k[cols].T)
    s[_mask(rows, cols, causal, kv_len, block_mask, block)] = -np.inf
    p = probabilities(s, _f64(lse))
    dp = do @ v[cols].T
    ds = p * (dp - _f64(d_row)[:, None])
    return {"dK": float(scale) * (ds.T @ q), "dV": p.T @ do}


def attention_forward(q, k, v, scale, causal=False, kv_len=None, rows=None, block_mask=None,
                      block=128):
    """(O[rows], LSE[rows]) of exact attention for one (batch, head) slice."""
    st = row_statistics(q, k, v, None, scale, causal, kv_len, rows, block_mask, block)
    return st["O"], st["LSE"]


def attention_backward(q, k, v, do, scale, causal=False, kv_len=None, block_mask=None, block=128):
    """Full forward + backward of one (batch, head) slice: dict with O, LSE, D, dQ, dK, dV."""
    st = row_statistics(q, k, v, do, scale, causal, kv_len, None, block_mask, block)
    kg = key_gradients(q, k, v, do, scale, st["LSE"], st["D"], causal, kv_len, None, None,
                       block_mask, block)
    st.update(kg)
    return st


def tiled_forward(q, k, v, scale, block, causal=False, kv_len=None, trace=None):
    """Online-softmax forward over key blocks of ``block`` keys, one query row at a time.

    State per row: running max m, running sum l (relative to m) and unnormalised output O~.
    For each key block: m~ = rowmax(S_ij), P~ = exp(S_ij - m~), l~ = rowsum(P~);
    m_new = max(m, m~); l_new = e^(m - m_new) l + e^(m~ - m_new) l~;
    O~_new = e^(m - m_new) O~ + e^(m~ - m_new) P~ V_j; finally O = O~ / l.
    Returns (O, LSE) with LSE = m + log(l).  ``trace`` (a list) receives, per row and block,
    the tuple (row, block, m~, l~, O~ of the block alone, m_new, l_new, O~_new) for tests.
    """
    q = _f64(q)
    v = _f64(v)
    n_q, n_k = q.shape[0], _f64(k).shape[0]
    out = np.zeros((n_q, v.shape[1]))
    lse = np.full(n_q, -np.inf)
    for i in range(n_q):
        s_row = masked_scores(q, k, scale, causal, kv_len, [i])[0]
        m, l, o_t = -np.inf, 0.0, np.zeros(v.shape[1])
        for b0 in range(0, n_k, block):
            s_blk = s_row[b0:b0 + block]
            m_blk = s_blk.max()
            if not np.isfinite(m_blk):
                continue  # every key of this block is masked: the block contributes nothing
            p_blk = np.exp(s_blk - m_blk)
            l_blk = p_blk.sum()
            o_blk = p_blk @ v[b0:b0 + block]
            m_new = max(m, m_blk)
            a = np.exp(m - m_new)  # 0 when m is still -inf
            b = np.exp(m_blk - m_new)
            l = a * l + b * l_blk
            o_t = a * o_t + b * o_blk
            m = m_new
            if trace is not None:
                trace.append((i, b0 // block, m_blk, l_blk, o_blk.copy(), m, l, o_t.copy()))
        if l > 0.0:
            out[i] = o_t / l
            lse[i] = m + np.log(l)
    return out, lse
