"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* the worked online-softmax example printed on the tutorial page (tests/golden/);
* closed forms: rows of P sum to one, identical keys give the mean of V, N = 1 gives V_0;
* invariances of the definition (shifting every key by one vector, adding a constant to V,
  permuting keys and values together);
* the softmax-backward identity D_i = dO_i . O_i (first page, 关键设计三) and sum_j dS_ij = 0;
* central finite differences of <dO, O> for the gradients;
* PyTorch's own CPU attention routine in float64 (a library routine, used here only as a
  check of the oracle).

Each pin is chosen so that a plausible slip in the oracle (a missing scale, a transposed
operand, a wrong mask index, a missing -D term) fails at least one of them.
"""

import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "online_softmax_worked_example.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, value, decimals = line.split()
            if "," in value:
                vals[name] = (np.array([float(x) for x in value.split(",")]), int(decimals))
            else:
                vals[name] = (float(value), int(decimals))
    return vals


def _close_printed(x, printed, decimals):
    # within one unit of the last printed decimal place
    return abs(x - printed) <= 10.0 ** (-decimals) * 1.0 + 1e-12


def _rand(n, d, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, d)) * sigma


# ---------------------------------------------------------------- worked example (tutorial page)

def test_worked_example_online_merge():
    g = _golden()
    scores = g["scores"][0]
    values = g["values"][0]
    block = int(g["block_size"][0])
    # one query row whose scaled scores are exactly `scores`: q = [1], k_j = [s_j], scale 1
    q = np.array([[1.0]])
    k = scores.reshape(-1, 1)
    v = values.reshape(-1, 1)
    trace = []
    o, lse = oracle.tiled_forward(q, k, v, scale=1.0, block=block, trace=trace)
    (_, _, m1, l1, ot1, _, _, _), (_, _, m2, l2, ot2, m, l, ot) = trace
    for name, got in [("m1", m1), ("l1", l1), ("m2", m2), ("l2", l2), ("m", m), ("l", l),
                      ("O_tilde1", ot1[0]), ("O_tilde2", ot2[0]), ("O_tilde", ot[0]),
                      ("O", o[0, 0])]:
        printed, dec = g[name]
        assert _close_printed(got, printed, dec), (name, got, printed)
    # the direct denominator the page computes with the global max
    printed, dec = g["l_direct"]
    assert _close_printed(np.exp(scores - scores.max()).sum(), printed, dec)
    # and the plain definition agrees with the recurrence to rounding
    o_def, lse_def = oracle.attention_forward(q, k, v, scale=1.0)
    assert abs(o_def[0, 0] - o[0, 0]) < 1e-12
    assert abs(lse_def[0] - lse[0]) < 1e-12
    assert abs(lse_def[0] - (m + np.log(l))) < 1e-12


# ---------------------------------------------------------------- forward closed forms

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kv_len", [None, 7])
def test_rows_of_p_sum_to_one(causal, kv_len):
    q, k = _rand(13, 5, 1), _rand(13, 5, 2)
    s = oracle.masked_scores(q, k, 0.7, causal, kv_len)
    p = oracle.probabilities(s, oracle.row_logsumexp(s))
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    assert np.all(p[np.isinf(s)] == 0.0)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
    if kv_len is not None:
        assert np.all(p[:, kv_len:] == 0.0)


def test_scale_enters_scores():
    q, k = _rand(4, 3, 3), _rand(6, 3, 4)
    s = oracle.masked_scores(q, k, 0.5)
    # element (i, j) by an explicit loop: 0.5 * sum_c q[i, c] k[j, c]
    for i in range(4):
        for j in range(6):
            assert abs(s[i, j] - 0.5 * sum(q[i, c] * k[j, c] for c in range(3))) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    n, d = 9, 4
    q = _rand(n, d, 5)
    k = np.tile(_rand(1, d, 6), (n, 1))
    v = _rand(n, d, 7)
    o, _ = oracle.attention_forward(q, k, v, scale=0.9, causal=causal)
    if causal:
        want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    else:
        want = np.tile(v.mean(axis=0), (n, 1))
    assert np.max(np.abs(o - want)) < 1e-12


def test_zero_scale_is_uniform():
    q, k, v = _rand(8, 4, 8), _rand(8, 4, 9), _rand(8, 4, 10)
    o, lse = oracle.attention_forward(q, k, v, scale=0.0)
    assert np.max(np.abs(o - v.mean(axis=0))) < 1e-12
    assert np.max(np.abs(lse - np.log(8.0))) < 1e-12


def test_single_key_and_causal_first_row():
    q, k, v = _rand(5, 4, 11), _rand(5, 4, 12), _rand(5, 4, 13)
    o, lse = oracle.attention_forward(q, k, v, scale=0.3, causal=True)
    assert np.max(np.abs(o[0] - v[0])) < 1e-14
    assert abs(lse[0] - 0.3 * q[0] @ k[0]) < 1e-14
    o1, lse1 = oracle.attention_forward(q[:1], k[:1], v[:1], scale=0.3)
    assert np.max(np.abs(o1[0] - v[0])) < 1e-14


def test_kv_len_one_gives_first_value():
    q, k, v = _rand(6, 4, 14), _rand(6, 4, 15), _rand(6, 4, 16)
    o, lse = oracle.attention_forward(q, k, v, scale=0.4, kv_len=1)
    assert np.max(np.abs(o - v[0])) < 1e-14
    assert np.max(np.abs(lse - 0.4 * q @ k[0])) < 1e-13


def test_fully_masked_row_convention():
    q, k, v, do = (_rand(4, 3, s) for s in (17, 18, 19, 20))
    st = oracle.attention_backward(q, k, v, do, scale=0.5, kv_len=0)
    assert np.all(st["O"] == 0.0) and np.all(np.isneginf(st["LSE"]))
    for name in ("dQ", "dK", "dV"):
        assert np.all(st[name] == 0.0) and not np.any(np.isnan(st[name]))


def test_shift_and_permutation_invariance():
    n, d = 10, 6
    q, k, v = _rand(n, d, 21), _rand(n, d, 22), _rand(n, d, 23)
    o, lse = oracle.attention_forward(q, k, v, scale=0.8)
    u = _rand(1, d, 24)
    o2, lse2 = oracle.attention_forward(q, k + u, v, scale=0.8)
    assert np.max(np.abs(o2 - o)) < 1e-12
    assert np.max(np.abs(lse2 - (lse + 0.8 * (q @ u.T)[:, 0]))) < 1e-12
    o3, _ = oracle.attention_forward(q, k, v + 2.5, scale=0.8)
    assert np.max(np.abs(o3 - (o + 2.5))) < 1e-12
    perm = np.random.default_rng(25).permutation(n)
    o4, lse4 = oracle.attention_forward(q, k[perm], v[perm], scale=0.8)
    assert np.max(np.abs(o4 - o)) < 1e-12 and np.max(np.abs(lse4 - lse)) < 1e-12


@pytest.mark.parametrize("causal,kv_len,block", [(False, None, 3), (True, None, 4),
                                                 (False, 9, 5), (True, 11, 2)])
def test_online_recurrence_equals_definition(causal, kv_len, block):
    n, d = 14, 5
    q, k, v = _rand(n, d, 26, 2.0), _rand(n, d, 27, 2.0), _rand(n, d, 28)
    o_t, lse_t = oracle.tiled_forward(q, k, v, 0.6, block, causal, kv_len)
    o, lse = oracle.attention_forward(q, k, v, 0.6, causal, kv_len)
    assert np.max(np.abs(o_t - o)) < 1e-12
    assert np.max(np.abs(lse_t - lse)) < 1e-12


def test_row_subset_matches_full():
    n, d = 12, 4
    q, k, v, do = (_rand(n, d, s) for s in (29, 30, 31, 32))
    full = oracle.row_statistics(q, k, v, do, 0.7, True, 10)
    rows = [0, 5, 11]
    sub = oracle.row_statistics(q, k, v, do, 0.7, True, 10, rows=rows)
    for name in ("O", "LSE", "D", "dQ"):
        assert np.max(np.abs(sub[name] - full[name][rows])) < 1e-13


# ---------------------------------------------------------------- backward

def test_d_identity_and_ds_rows_sum_to_zero():
    n, d = 11, 5
    q, k, v, do = (_rand(n, d, s) for s in (33, 34, 35, 36))
    st = oracle.attention_backward(q, k, v, do, 0.45, causal=True)
    # D_i = sum_j P_ij dP_ij equals dO_i . O_i
    assert np.max(np.abs(st["D"] - (do * st["O"]).sum(axis=1))) < 1e-12
    s = oracle.masked_scores(q, k, 0.45, causal=True)
    p = oracle.probabilities(s, st["LSE"])
    ds = p * (do @ v.T - st["D"][:, None])
    assert np.max(np.abs(ds.sum(axis=1))) < 1e-12
    # sum_j dV_j = sum_i dO_i (rows of P sum to one)
    assert np.max(np.abs(st["dV"].sum(axis=0) - do.sum(axis=0))) < 1e-12


def _loss(q, k, v, do, scale, causal, kv_len):
    o, _ = oracle.attention_forward(q, k, v, scale, causal, kv_len)
    return float((o * do).sum())


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 4), (True, 5)])
def test_gradients_match_finite_differences(causal, kv_len):
    n, d, scale, h = 6, 4, 0.7, 1e-6
    q, k, v, do = (_rand(n, d, s) for s in (37, 38, 39, 40))
    st = oracle.attention_backward(q, k, v, do, scale, causal, kv_len)
    for name, x in (("dQ", q), ("dK", k), ("dV", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"dQ": (xp, k, v), "dK": (q, xp, v), "dV": (q, k, xp)}[name]
            argm = {"dQ": (xm, k, v), "dK": (q, xm, v), "dV": (q, k, xm)}[name]
            num[idx] = (_loss(*args, do, scale, causal, kv_len) - _loss(*argm, do, scale, causal, kv_len)) / (2 * h)
        err = np.linalg.norm(num - st[name]) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-7, (name, err)
    if kv_len is not None:
        assert np.all(st["dK"][kv_len:] == 0.0) and np.all(st["dV"][kv_len:] == 0.0)


def test_key_subset_matches_full():
    n, d = 10, 3
    q, k, v, do = (_rand(n, d, s) for s in (41, 42, 43, 44))
    st = oracle.attention_backward(q, k, v, do, 0.9, True, 8)
    cols = [1, 7, 9]
    kg = oracle.key_gradients(q, k, v, do, 0.9, st["LSE"], st["D"], True, 8, cols)
    assert np.max(np.abs(kg["dK"] - st["dK"][cols])) < 1e-13
    assert np.max(np.abs(kg["dV"] - st["dV"][cols])) < 1e-13


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 13)])
def test_against_torch_cpu_attention_float64(causal, kv_len):
    n, d, scale = 17, 8, 0.35
    q, k, v, do = (_rand(n, d, s, 2.0) for s in (45, 46, 47, 48))
    st = oracle.attention_backward(q, k, v, do, scale, causal, kv_len)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = torch.ones(n, n, dtype=torch.bool)
    if causal:
        mask &= torch.tril(torch.ones(n, n, dtype=torch.bool))
    if kv_len is not None:
        mask[:, kv_len:] = False
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=mask, scale=scale)[0, 0]
    o.backward(torch.tensor(do))
    assert np.max(np.abs(o.detach().numpy() - st["O"])) < 1e-12
    for name, t in (("dQ", tq), ("dK", tk), ("dV", tv)):
        assert np.max(np.abs(t.grad.numpy() - st[name])) < 1e-11, name


def test_key_gradients_sum_over_row_partition():
    n, d = 12, 3
    q, k, v, do = (_rand(n, d, s) for s in (49, 50, 51, 52))
    st = oracle.attention_backward(q, k, v, do, 0.6, True, 10)
    parts = [np.arange(0, 5), np.arange(5, 12)]
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for rows in parts:
        kg = oracle.key_gradients(q, k, v, do, 0.6, st["LSE"][rows], st["D"][rows], True, 10,
                                  rows=rows)
        dk += kg["dK"]
        dv += kg["dV"]
    assert np.max(np.abs(dk - st["dK"])) < 1e-13 and np.max(np.abs(dv - st["dV"])) < 1e-13


# ---------------------------------------------------------------- block mask (block-sparse)


def _expand(bm, block, n):
    """Element mask of a block mask, written independently of the oracle (Kronecker product)."""
    return np.kron(np.asarray(bm, dtype=np.int64), np.ones((block, block), dtype=np.int64))[:n, :n] != 0


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 14), (True, 15)])
def test_block_mask_against_torch_cpu_attention_float64(causal, kv_len):
    n, d, scale, block = 19, 8, 0.4, 4
    q, k, v, do = (_rand(n, d, s, 1.5) for s in (61, 62, 63, 64))
    rng = np.random.default_rng(65)
    nb = -(-n // block)
    bm = (rng.random((nb, nb)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)  # every row keeps at least its diagonal block
    bm[:, 0] = 1             # ... and key block 0, so that kv_len never empties a row
    st = oracle.attention_backward(q, k, v, do, scale, causal, kv_len, block_mask=bm, block=block)
    mask = torch.tensor(_expand(bm, block, n))
    if causal:
        mask &= torch.tril(torch.ones(n, n, dtype=torch.bool))
    if kv_len is not None:
        mask[:, kv_len:] = False
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=mask, scale=scale)[0, 0]
    o.backward(torch.tensor(do))
    assert np.max(np.abs(o.detach().numpy() - st["O"])) < 1e-12
    for name, t in (("dQ", tq), ("dK", tk), ("dV", tv)):
        assert np.max(np.abs(t.grad.numpy() - st[name])) < 1e-11, name


def test_block_diagonal_mask_is_independent_attention_per_block():
    n, d, scale, block = 12, 3, 0.8, 4
    q, k, v, do = (_rand(n, d, s) for s in (66, 67, 68, 69))
    bm = np.eye(3, dtype=np.uint8)
    st = oracle.attention_backward(q, k, v, do, scale, block_mask=bm, block=block)
    for b0 in range(0, n, block):
        sl = slice(b0, b0 + block)
        ref = oracle.attention_backward(q[sl], k[sl], v[sl], do[sl], scale)
        for name in ("O", "LSE", "dQ", "dK", "dV"):
            assert np.max(np.abs(st[name][sl] - ref[name])) < 1e-13, name


def test_zero_block_equals_removed_keys():
    n, d, scale, block = 9, 4, 0.6, 3
    q, k, v, do = (_rand(n, d, s) for s in (70, 71, 72, 73))
    bm = np.ones((3, 3), dtype=np.uint8)
    bm[1, 2] = 0  # query rows 3..5 do not see keys 6..8
    o, lse = oracle.attention_forward(q, k, v, scale, block_mask=bm, block=block)
    keep = np.r_[0:6]
    o_ref, lse_ref = oracle.attention_forward(q[3:6], k[keep], v[keep], scale)
    assert np.max(np.abs(o[3:6] - o_ref)) < 1e-13 and np.max(np.abs(lse[3:6] - lse_ref)) < 1e-13
    o_full, _ = oracle.attention_forward(q, k, v, scale)
    rows = np.r_[0:3, 6:9]
    assert np.array_equal(o[rows], o_full[rows])  # other rows keep every key: unchanged


def test_all_ones_block_mask_is_dense_and_empty_row_is_zero():
    n, d, scale, block = 10, 4, 0.5, 4
    q, k, v, do = (_rand(n, d, s) for s in (74, 75, 76, 77))
    dense = oracle.attention_backward(q, k, v, do, scale, True, 9)
    ones = oracle.attention_backward(q, k, v, do, scale, True, 9, block_mask=np.ones((3, 3)), block=block)
    for name in ("O", "LSE", "dQ", "dK", "dV"):
        assert np.array_equal(dense[name], ones[name]), name
    bm = np.ones((3, 3), dtype=np.uint8)
    bm[1, :] = 0  # rows 4..7 keep no block
    st = oracle.attention_backward(q, k, v, do, scale, block_mask=bm, block=block)
    assert np.all(st["O"][4:8] == 0) and np.all(st["LSE"][4:8] == -np.inf)
    assert np.all(st["dQ"][4:8] == 0)
    # the other rows' gradients are those of attention without rows 4..7
    rows = np.r_[0:4, 8:10]
    ref = oracle.attention_backward(q[rows], k, v, do[rows], scale)
    assert np.max(np.abs(st["dK"] - ref["dK"])) < 1e-13 and np.max(np.abs(st["dV"] - ref["dV"])) < 1e-13


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, 5)])
def test_block_mask_gradients_match_finite_differences(causal, kv_len):
    n, d, scale, h, block = 6, 3, 0.7, 1e-6, 2
    q, k, v, do = (_rand(n, d, s) for s in (78, 79, 80, 81))
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]], dtype=np.uint8)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward(qq, kk, vv, scale, causal, kv_len, block_mask=bm, block=block)
        return float((o * do).sum())

    st = oracle.attention_backward(q, k, v, do, scale, causal, kv_len, block_mask=bm, block=block)
    for name, x in (("dQ", q), ("dK", k), ("dV", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            pick = {"dQ": lambda y: (y, k, v), "dK": lambda y: (q, y, v), "dV": lambda y: (q, k, y)}[name]
            num[idx] = (loss(*pick(xp)) - loss(*pick(xm))) / (2 * h)
        err = np.linalg.norm(num - st[name]) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-7, (name, err)
