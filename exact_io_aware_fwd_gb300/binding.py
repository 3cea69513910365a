"""Thin ctypes binding of libfa_sm103.so with the C-ABI's names.

Only argument marshalling happens here (torch tensors -> device pointers, the current CUDA
stream, output/workspace allocation through torch's caching allocator).  Every step of the
computation runs in the library's CUDA kernels; there is no fallback of any kind: if the
library is missing or the device is not an sm_103 GPU (GB300) the call raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from .build_lib import LIB_PATH

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5

EXPORTED = [
    "fa_fwd",
    "fa_bwd_workspace_size",
    "fa_bwd",
    "fa_bwd_preprocess",
    "fa_bwd_dkdv",
    "fa_bwd_dq_convert",
    "fa_bwd_noalloc",
    "fa_bwd_deterministic",
    "fa_fwd_gqa",
    "fa_bwd_gqa",
    "fa_fwd_varlen",
    "fa_bwd_varlen_workspace_size",
    "fa_bwd_varlen",
    "fa_block_index_size",
    "fa_block_index_build",
    "fa_fwd_block_sparse",
    "fa_bwd_block_sparse",
    "fa_get_error",
    "fa_status_string",
]

_lib = None


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of libfa_sm103.so."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp, sz, vp]
    lib.fa_bwd_preprocess.restype = i
    lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, sz, vp]
    lib.fa_bwd_dkdv.restype = i
    lib.fa_bwd_dq_convert.argtypes = [vp, i, i, i, i, f, vp, sz, vp]
    lib.fa_bwd_dq_convert.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                          vp, vp, sz, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp]
    lib.fa_fwd_gqa.restype = i
    lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, i,
                               vp, sz, vp]
    lib.fa_bwd_gqa.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f,
                                  i, vp, sz, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_block_index_size.argtypes = [i, i]
    lib.fa_block_index_size.restype = sz
    lib.fa_block_index_build.argtypes = [vp, i, i, vp, sz, vp]
    lib.fa_block_index_build.restype = i
    lib.fa_fwd_block_sparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp, i, vp]
    lib.fa_fwd_block_sparse.restype = i
    lib.fa_bwd_block_sparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                         vp, vp, i, i, vp, sz, vp]
    lib.fa_bwd_block_sparse.restype = i
    lib.fa_get_error.argtypes = [vp]
    lib.fa_get_error.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def _check(status, where):
    if status != FA_OK:
        raise FAError(status, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_qkv(*ts):
    ref = ts[0]
    if ref.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous CUDA bfloat16 tensors")
        if t.shape != ref.shape:
            raise ValueError("shape mismatch")
        if t.device != ref.device:
            raise ValueError("tensors on different devices")
    return tuple(ref.shape)


def _want(t, shape, dtype, device, name):
    """`t` itself after checking that the library may write or read it as a dense array of
    `shape`: a contiguous `dtype` tensor on `device` (the kernels address it by pointer only)."""
    if (not isinstance(t, torch.Tensor) or t.device != device or t.dtype != dtype
            or not t.is_contiguous() or tuple(t.shape) != tuple(shape)):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"on {device}")
    return t


def _out(t, shape, dtype, device, name):
    """A new output tensor, or the caller's after the checks of `_want`."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _want(t, shape, dtype, device, name)


def _workspace(ws, nbytes, device):
    """(tensor, size in bytes) of the backward workspace: a new byte array, or the caller's
    contiguous tensor on `device` (any dtype; its size is counted in bytes)."""
    if ws is None:
        return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device), max(int(nbytes), 1)
    if not isinstance(ws, torch.Tensor) or ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    return ws, ws.numel() * ws.element_size()


def _kv(kv_lens, B, device):
    if kv_lens is None:
        return None
    kv = kv_lens.to(device=device, dtype=torch.int32).contiguous()
    if kv.numel() != B:
        raise ValueError("kv_lens must have B entries")
    return kv


def _scale(scale):
    return -1.0 if scale is None else float(scale)


def fa_fwd(q, k, v, causal=False, scale=None, kv_lens=None, out=None, lse=None, stream=None):
    """O, LSE = exact attention of [B,H,N,d] bf16 q, k, v (see include/fa.h)."""
    B, H, N, d = _check_qkv(q, k, v)
    out = _out(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                               int(bool(causal)), _scale(scale), _ptr(kv), _stream(stream))
    _check(st, "fa_fwd")
    return out, lse


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def workspace_for(q):
    B, H, N, d = q.shape
    nbytes = fa_bwd_workspace_size(B, H, N, d)
    if nbytes == 0:
        raise FAError(FA_ERR_INVALID_ARG, "fa_bwd_workspace_size")
    # torch's allocator returns 512-byte aligned blocks
    return torch.empty(nbytes, device=q.device, dtype=torch.uint8)


def fa_bwd(q, k, v, o, do, lse, causal=False, scale=None, kv_lens=None, dq=None, dk=None,
           dv=None, workspace=None, stream=None):
    """dQ, dK, dV of exact attention given the forward's O and LSE (see include/fa.h)."""
    B, H, N, d = _check_qkv(q, k, v, o, do)
    _want(lse, (B, H, N), torch.float32, q.device, "lse")
    dq, dk, dv = (_out(t, q.shape, torch.bfloat16, q.device, n)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    ws, ws_bytes = _workspace(workspace, fa_bwd_workspace_size(B, H, N, d), q.device)
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                               _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), _scale(scale),
                               _ptr(kv), _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "fa_bwd")
    return dq, dk, dv


def fa_bwd_deterministic(q, k, v, o, do, lse, causal=False, scale=None, kv_lens=None, dq=None,
                         dk=None, dv=None, workspace=None, stream=None):
    """fa_bwd with run-to-run bit-identical results (dQ without atomics; see include/fa.h)."""
    B, H, N, d = _check_qkv(q, k, v, o, do)
    _want(lse, (B, H, N), torch.float32, q.device, "lse")
    dq, dk, dv = (_out(t, q.shape, torch.bfloat16, q.device, n)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    ws, ws_bytes = _workspace(workspace, fa_bwd_workspace_size(B, H, N, d), q.device)
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do),
                                             _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                             int(bool(causal)), _scale(scale), _ptr(kv), _ptr(ws),
                                             ws_bytes, _stream(stream))
    _check(st, "fa_bwd_deterministic")
    return dq, dk, dv


def fa_bwd_preprocess(o, do, lse, workspace, stream=None):
    B, H, N, d = _check_qkv(o, do)
    _want(lse, (B, H, N), torch.float32, o.device, "lse")
    ws, ws_bytes = _workspace(workspace, 0, o.device)
    st = load_library().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), B, H, N, d,
                                          _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "fa_bwd_preprocess")


def fa_bwd_dkdv(q, k, v, do, dk, dv, workspace, causal=False, scale=None, kv_lens=None,
                stream=None):
    B, H, N, d = _check_qkv(q, k, v, do, dk, dv)
    kv = _kv(kv_lens, B, q.device)
    ws, ws_bytes = _workspace(workspace, 0, q.device)
    st = load_library().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), B,
                                    H, N, d, int(bool(causal)), _scale(scale), _ptr(kv),
                                    _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "fa_bwd_dkdv")


def fa_bwd_dq_convert(dq, workspace, scale=None, stream=None):
    B, H, N, d = _check_qkv(dq)
    ws, ws_bytes = _workspace(workspace, 0, dq.device)
    st = load_library().fa_bwd_dq_convert(_ptr(dq), B, H, N, d, _scale(scale), _ptr(ws),
                                          ws_bytes, _stream(stream))
    _check(st, "fa_bwd_dq_convert")


def fa_bwd_noalloc(q, k, v, o, do, lse, causal=False, scale=None, kv_lens=None, dq=None,
                   dk=None, dv=None, stream=None):
    """fa_bwd with the library's static workspace, for callers that cannot allocate device
    memory (see include/fa.h); calls that overlap on the GPU must be serialised."""
    B, H, N, d = _check_qkv(q, k, v, o, do)
    _want(lse, (B, H, N), torch.float32, q.device, "lse")
    dq, dk, dv = (_out(t, q.shape, torch.bfloat16, q.device, n)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                       _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                       int(bool(causal)), _scale(scale), _ptr(kv),
                                       _stream(stream))
    _check(st, "fa_bwd_noalloc")
    return dq, dk, dv


def fa_get_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status."""
    return int(load_library().fa_get_error(_stream(stream)))


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


class BlockIndex:
    """Device block-sparse index built from a uint8 block mask over 128 x 128 tiles."""

    def __init__(self, tensor, N, mask_heads):
        self.tensor, self.N, self.mask_heads = tensor, N, mask_heads


def fa_block_index_size(N, mask_heads=1) -> int:
    return int(load_library().fa_block_index_size(int(N), int(mask_heads)))


def fa_block_index_build(block_mask, N, stream=None) -> BlockIndex:
    """Index of a [T, T] or [mask_heads, T, T] mask (T = ceil(N / 128), nonzero = kept)."""
    if not block_mask.is_cuda:
        raise ValueError("block_mask must be a CUDA tensor")
    T = (int(N) + 127) // 128
    m = block_mask.to(torch.uint8).contiguous()
    if m.dim() == 2:
        m = m[None]
    if m.dim() != 3 or m.shape[1:] != (T, T):
        raise ValueError(f"block_mask must be [T, T] or [heads, T, T] with T = {T}")
    heads = m.shape[0]
    nbytes = fa_block_index_size(N, heads)
    idx = torch.empty(nbytes // 4, dtype=torch.int32, device=m.device)
    st = load_library().fa_block_index_build(_ptr(m), int(N), heads, _ptr(idx), nbytes,
                                             _stream(stream))
    _check(st, "fa_block_index_build")
    return BlockIndex(idx, int(N), heads)


def fa_fwd_block_sparse(q, k, v, index: BlockIndex, causal=False, scale=None, kv_lens=None,
                        out=None, lse=None, stream=None):
    """fa_fwd restricted to the kept 128 x 128 tiles of `index` (see include/fa.h)."""
    B, H, N, d = _check_qkv(q, k, v)
    if index.N != N:
        raise ValueError("block index built for another N")
    if index.tensor.device != q.device:
        raise ValueError("block index on another device")
    out = _out(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_fwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                            N, d, int(bool(causal)), _scale(scale), _ptr(kv),
                                            _ptr(index.tensor), index.mask_heads, _stream(stream))
    _check(st, "fa_fwd_block_sparse")
    return out, lse


def fa_bwd_block_sparse(q, k, v, o, do, lse, index: BlockIndex, causal=False, scale=None,
                        kv_lens=None, deterministic=False, dq=None, dk=None, dv=None,
                        workspace=None, stream=None):
    """fa_bwd restricted to the kept tiles of `index` (see include/fa.h)."""
    B, H, N, d = _check_qkv(q, k, v, o, do)
    if index.N != N:
        raise ValueError("block index built for another N")
    if index.tensor.device != q.device:
        raise ValueError("block index on another device")
    _want(lse, (B, H, N), torch.float32, q.device, "lse")
    dq, dk, dv = (_out(t, q.shape, torch.bfloat16, q.device, n)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    ws, ws_bytes = _workspace(workspace, fa_bwd_workspace_size(B, H, N, d), q.device)
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_bwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do),
                                            _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                            int(bool(causal)), _scale(scale), _ptr(kv),
                                            _ptr(index.tensor), index.mask_heads,
                                            int(bool(deterministic)), _ptr(ws), ws_bytes,
                                            _stream(stream))
    _check(st, "fa_bwd_block_sparse")
    return dq, dk, dv


def _check_group(q, k):
    """(B, H, Hkv, N, d) of [B, H, N, d] queries and [B, Hkv, N, d] keys."""
    for t in (q, k):
        if t.dim() != 4 or not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous CUDA bfloat16 [B, heads, N, d] tensors")
    B, H, N, d = q.shape
    if k.shape[0] != B or k.shape[2:] != (N, d) or H % k.shape[1] != 0:
        raise ValueError("K must be [B, Hkv, N, d] with H % Hkv == 0")
    if k.device != q.device:
        raise ValueError("tensors on different devices")
    return B, H, k.shape[1], N, d


def fa_fwd_gqa(q, k, v, causal=False, scale=None, kv_lens=None, out=None, lse=None, stream=None):
    """Grouped-query forward: q [B, H, N, d], k and v [B, Hkv, N, d] (see include/fa.h)."""
    B, H, Hkv, N, d = _check_group(q, k)
    _want(v, k.shape, torch.bfloat16, q.device, "v")
    out = _out(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N,
                                   d, int(bool(causal)), _scale(scale), _ptr(kv), _stream(stream))
    _check(st, "fa_fwd_gqa")
    return out, lse


def fa_bwd_gqa(q, k, v, o, do, lse, causal=False, scale=None, kv_lens=None, deterministic=False,
               dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Grouped-query backward; dK, dV [B, Hkv, N, d] sum over each key/value head's group."""
    B, H, Hkv, N, d = _check_group(q, k)
    _want(v, k.shape, torch.bfloat16, q.device, "v")
    _want(o, q.shape, torch.bfloat16, q.device, "o")
    _want(do, q.shape, torch.bfloat16, q.device, "do")
    _want(lse, (B, H, N), torch.float32, q.device, "lse")
    dq = _out(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out(dv, k.shape, torch.bfloat16, q.device, "dv")
    ws, ws_bytes = _workspace(workspace, fa_bwd_workspace_size(B, H, N, d), q.device)
    kv = _kv(kv_lens, B, q.device)
    st = load_library().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d,
                                   int(bool(causal)), _scale(scale), _ptr(kv),
                                   int(bool(deterministic)), _ptr(ws), ws_bytes,
                                   _stream(stream))
    _check(st, "fa_bwd_gqa")
    return dq, dk, dv


def _check_packed(q, k, cu_seqlens):
    for t in (q, k):
        if t.dim() != 3 or not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous CUDA bfloat16 [total, heads, d] tensors")
    total, H, d = q.shape
    if k.shape[0] != total or k.shape[2] != d or H % k.shape[1] != 0:
        raise ValueError("K must be [total, Hkv, d] with H % Hkv == 0")
    if (cu_seqlens.dtype != torch.int32 or cu_seqlens.device != q.device
            or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2 or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 vector of B + 1 offsets on "
                         "q's device")
    if k.device != q.device:
        raise ValueError("tensors on different devices")
    return total, H, k.shape[1], d, cu_seqlens.numel() - 1


def fa_bwd_varlen_workspace_size(B, total, H, d) -> int:
    return int(load_library().fa_bwd_varlen_workspace_size(int(B), int(total), int(H), int(d)))


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, scale=None, out=None, lse=None,
                  stream=None):
    """Packed variable-length forward: q [total, H, d], k and v [total, Hkv, d], LSE [H, total]."""
    total, H, Hkv, d, B = _check_packed(q, k, cu_seqlens)
    _want(v, k.shape, torch.bfloat16, q.device, "v")
    out = _out(out, q.shape, torch.bfloat16, q.device, "out")
    lse = _out(lse, (H, total), torch.float32, q.device, "lse")
    st = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                      _ptr(cu_seqlens), B, int(max_seqlen), total, H, Hkv, d,
                                      int(bool(causal)), _scale(scale), _stream(stream))
    _check(st, "fa_fwd_varlen")
    return out, lse


def fa_bwd_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen, causal=False, scale=None,
                  deterministic=False, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Packed variable-length backward (see include/fa.h)."""
    total, H, Hkv, d, B = _check_packed(q, k, cu_seqlens)
    _want(v, k.shape, torch.bfloat16, q.device, "v")
    _want(o, q.shape, torch.bfloat16, q.device, "o")
    _want(do, q.shape, torch.bfloat16, q.device, "do")
    _want(lse, (H, total), torch.float32, q.device, "lse")
    dq = _out(dq, q.shape, torch.bfloat16, q.device, "dq")
    dk = _out(dk, k.shape, torch.bfloat16, q.device, "dk")
    dv = _out(dv, k.shape, torch.bfloat16, q.device, "dv")
    workspace, ws_bytes = _workspace(workspace, fa_bwd_varlen_workspace_size(B, total, H, d),
                                     q.device)
    st = load_library().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens), B,
                                      int(max_seqlen), total, H, Hkv, d, int(bool(causal)),
                                      _scale(scale), int(bool(deterministic)), _ptr(workspace),
                                      ws_bytes, _stream(stream))
    _check(st, "fa_bwd_varlen")
    return dq, dk, dv

