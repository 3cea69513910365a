"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, run the fp64
oracle on the same (bf16-rounded) inputs, and compare with the stated tolerances:

  O    max-abs error <= 1e-2 (before the output's bf16 rounding, see compare_slice) and
       relative Frobenius error <= 5e-3
  LSE  max-abs error <= 1e-3
  dQ, dK, dV  relative Frobenius error <= 2e-2
(bf16 inputs and outputs, fp32 accumulation on the GPU).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_O_ABS = 1e-2
TOL_O_REL = 5e-3
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2
TOL_ZERO_GRAD = 1e-4  # absolute, where the exact gradient is identically zero

ROW_CHUNK = 2048


def run_gpu(q, k, v, do, causal, scale, kv_lens, with_bwd=True, deterministic=False,
            block_mask=None):
    """fa_fwd (+ fa_bwd, or fa_bwd_deterministic) on cuda:0; returns device tensors.  With a
    block mask (uint8 [T, T] or [H, T, T]) the block-sparse entry points run instead."""
    import exact_io_aware_fwd_gb300 as fa

    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    kv = kv_lens.to(dev) if kv_lens is not None else None
    if block_mask is not None:
        index = fa.fa_block_index_build(block_mask.to(dev), q.shape[2])
        o, lse = fa.fa_fwd_block_sparse(qd, kd, vd, index, causal=causal, scale=scale, kv_lens=kv)
    else:
        o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, scale=scale, kv_lens=kv)
    out = {"O": o, "LSE": lse}
    if with_bwd:
        dod = do.to(dev)
        if block_mask is not None:
            dq, dk, dv = fa.fa_bwd_block_sparse(qd, kd, vd, o, dod, lse, index, causal=causal,
                                                scale=scale, kv_lens=kv,
                                                deterministic=deterministic)
        else:
            bwd = fa.fa_bwd_deterministic if deterministic else fa.fa_bwd
            dq, dk, dv = bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale, kv_lens=kv)
        out.update(dQ=dq, dK=dk, dV=dv)
    st = fa.fa_get_error()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return out


def oracle_slice(q, k, v, do, causal, scale, kv_len, with_bwd=True, block_mask=None):
    """Full fp64 oracle outputs of one [N, d] slice, computed in row / key chunks."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    do = np.asarray(do, dtype=np.float64) if with_bwd else None
    n = q.shape[0]
    parts = []
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK))
        parts.append(oracle.row_statistics(q, k, v, do, scale, causal, kv_len, rows, block_mask))
    res = {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}
    if with_bwd:
        dk, dv = [], []
        for c0 in range(0, n, ROW_CHUNK):
            cols = np.arange(c0, min(n, c0 + ROW_CHUNK))
            kg = oracle.key_gradients(q, k, v, do, scale, res["LSE"], res["D"], causal, kv_len, cols,
                                      None, block_mask)
            dk.append(kg["dK"])
            dv.append(kg["dV"])
        res["dK"] = np.concatenate(dk)
        res["dV"] = np.concatenate(dv)
    return res


def bf16_half_ulp(x):
    """Half the spacing of bfloat16 numbers (8 significant bits) around |x|."""
    x = np.maximum(np.abs(x), np.finfo(np.float64).tiny)
    return np.ldexp(1.0, np.floor(np.log2(x)).astype(np.int64) - 8)


def f64(t):
    return t.detach().double().cpu().numpy()


def compare_slice(gpu_slice: dict, ref: dict, label: str, with_bwd=True, grad_tol=None):
    """Assert the tolerances on one (b, h) slice; returns the error figures."""
    errs = {}
    o = gpu_slice["O"]
    o_ref = ref["O"]
    errs["O_abs"] = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    nrm = np.linalg.norm(o_ref)
    errs["O_rel"] = float(np.linalg.norm(o - o_ref) / nrm) if nrm > 0 else float(np.linalg.norm(o))
    lse, lse_ref = gpu_slice["LSE"], ref["LSE"]
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), finite), f"{label}: LSE finiteness differs"
    assert np.all(lse[~finite] == lse_ref[~finite]), f"{label}: LSE of key-less rows"
    errs["LSE_abs"] = float(np.max(np.abs(lse[finite] - lse_ref[finite]))) if finite.any() else 0.0
    # O is returned in bf16: the 1e-2 bound applies to the value before that final rounding, so
    # each element may additionally differ by half a bf16 ulp of (|O_ref| + 1e-2).
    excess = np.abs(o - o_ref) - (TOL_O_ABS + bf16_half_ulp(np.abs(o_ref) + TOL_O_ABS))
    errs["O_abs_excess"] = float(np.max(excess)) if o.size else -1.0
    assert errs["O_abs_excess"] <= 0.0, (label, errs)
    assert errs["O_rel"] <= TOL_O_REL, (label, errs)
    assert errs["LSE_abs"] <= TOL_LSE, (label, errs)
    if with_bwd:
        for name in ("dQ", "dK", "dV"):
            g, r = gpu_slice[name], ref[name]
            assert np.all(np.isfinite(g)), f"{label}: non-finite {name}"
            nrm = np.linalg.norm(r)
            if nrm == 0:
                # the exact gradient vanishes (e.g. a single visible key: dS = P (dP - D) = 0);
                # the GPU's dP and D are rounded differently, so allow rounding-level residue
                errs[name] = float(np.max(np.abs(g)))
                assert errs[name] <= TOL_ZERO_GRAD, (label, name, errs)
            else:
                errs[name] = float(np.linalg.norm(g - r) / nrm)
                assert errs[name] <= (grad_tol or TOL_GRAD_REL), (label, name, errs)
    return errs


def check_case(q, k, v, do, causal, scale, kv_lens, slices=None, with_bwd=True, label="",
               grad_tol=None, deterministic=False, block_mask=None):
    """Run the CUDA path on the whole batch and compare the chosen (b, h) slices."""
    B, H, N, d = q.shape
    sc = (1.0 / d ** 0.5) if scale is None else scale
    out = run_gpu(q, k, v, do, causal, scale, kv_lens, with_bwd, deterministic, block_mask)
    torch.cuda.synchronize()
    slices = slices if slices is not None else [(b, h) for b in range(B) for h in range(H)]
    all_errs = []
    for b, h in slices:
        kv_len = int(kv_lens[b]) if kv_lens is not None else None
        ref = oracle_slice(q[b, h].float().numpy(), k[b, h].float().numpy(), v[b, h].float().numpy(),
                           do[b, h].float().numpy() if with_bwd else None, causal, sc, kv_len,
                           with_bwd, _head_mask(block_mask, h))
        got = {name: f64(t[b, h]) for name, t in out.items()}
        all_errs.append(compare_slice(got, ref, f"{label} b={b} h={h}", with_bwd, grad_tol))
    return out, all_errs


def _head_mask(block_mask, h):
    """The [T, T] numpy block mask of head h (None without a mask)."""
    if block_mask is None:
        return None
    m = block_mask.cpu().numpy()
    return m if m.ndim == 2 else m[h]



def compare_grad(g, r, label, tol=None):
    """Relative Frobenius error of one gradient (or the zero-gradient bound), asserted."""
    assert np.all(np.isfinite(g)), f"{label}: non-finite"
    nrm = np.linalg.norm(r)
    if nrm == 0:
        err = float(np.max(np.abs(g))) if g.size else 0.0
        assert err <= TOL_ZERO_GRAD, (label, err)
    else:
        err = float(np.linalg.norm(g - r) / nrm)
        assert err <= (tol or TOL_GRAD_REL), (label, err)
    return err


def check_heads(q_h, k_g, v_g, do_h, out_h, causal, scale, kv_len, label, grad_tol=None):
    """One key/value head and its group of query heads.

    q_h, do_h: lists (one per query head of the group) of [n, d] CPU bf16 slices; k_g, v_g: the
    group's [n, d] key/value slices; out_h: list of dicts of GPU results for those query heads
    (O, LSE, dQ as CPU float64) plus "dK", "dV" of the key/value head.  The oracle runs per
    query head; dK and dV of the shared head are the sums over the group (the chain rule for a
    shared input)."""
    k_np, v_np = k_g.float().numpy(), v_g.float().numpy()
    dk_ref = dv_ref = None
    for qq, dd, got in zip(q_h, do_h, out_h):
        ref = oracle_slice(qq.float().numpy(), k_np, v_np, dd.float().numpy(), causal, scale,
                           kv_len, True)
        fwd = {"O": got["O"], "LSE": got["LSE"]}
        compare_slice(fwd, ref, label, with_bwd=False)
        compare_grad(got["dQ"], ref["dQ"], label + " dQ", grad_tol)
        dk_ref = ref["dK"] if dk_ref is None else dk_ref + ref["dK"]
        dv_ref = ref["dV"] if dv_ref is None else dv_ref + ref["dV"]
    compare_grad(out_h[0]["dK"], dk_ref, label + " dK", grad_tol)
    compare_grad(out_h[0]["dV"], dv_ref, label + " dV", grad_tol)
