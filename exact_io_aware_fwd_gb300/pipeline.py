"""Host-resident forward + backward with copies overlapped with compute.

``attention_fwd_bwd_host`` is the call for data that lives in (pinned) host memory: it splits the
work into chunks of whole heads, and for each chunk copies Q, K, V, dO in on one stream, runs
fa_fwd and fa_bwd on a second and copies O, LSE, dQ, dK, dV out on a third, with CUDA events
ordering the three.  Chunks are independent (attention never mixes heads), so while chunk c
computes, chunk c+1 is copied in and chunk c-1 copied out.  Only orchestration happens here; the
arithmetic is the library's kernels.
"""

from __future__ import annotations

import torch

from . import binding


def _chunks(B, H, target=8, heads_per_chunk=None):
    """(b0, b1, h0, h1) pieces, each a contiguous slice q[b0:b1, h0:h1] of a [B, H, N, d] tensor:
    about `target` pieces of whole batches when B >= target, otherwise head ranges of one batch
    (`heads_per_chunk` overrides the head-range width)."""
    if heads_per_chunk is None and B >= target:
        per = -(-B // target)
        for b0 in range(0, B, per):
            yield b0, min(B, b0 + per), 0, H
        return
    if heads_per_chunk is None:
        heads_per_chunk = max(1, -(-(B * H) // target))
    heads_per_chunk = min(heads_per_chunk, H)
    for b in range(B):
        for h0 in range(0, H, heads_per_chunk):
            yield b, b + 1, h0, min(H, h0 + heads_per_chunk)


class HostAttention:
    """Device buffers, streams and events for repeated host-to-host fwd + bwd of one shape."""

    def __init__(self, B, H, N, d, device=None, heads_per_chunk=None):
        self.shape = (B, H, N, d)
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        dev = self.device
        mk = lambda: torch.empty(self.shape, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.q, self.k, self.v, self.do = mk(), mk(), mk(), mk()
        self.o, self.dq, self.dk, self.dv = mk(), mk(), mk(), mk()
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.kv = torch.empty((B,), dtype=torch.int32, device=dev)
        self.plan = list(_chunks(B, H, heads_per_chunk=heads_per_chunk))
        max_heads = max((b1 - b0) * (h1 - h0) for b0, b1, h0, h1 in self.plan)
        # chunks compute one after another on one stream, so one workspace serves them all
        self.workspace = torch.empty(binding.fa_bwd_workspace_size(1, max_heads, N, d),
                                     dtype=torch.uint8, device=dev)
        self.s_in = torch.cuda.Stream(dev)
        self.s_comp = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)

    def run(self, q, k, v, do, causal=False, scale=None, kv_lens=None, out=None,
            deterministic=False, block_index=None):
        """Host tensors in -> host tensors (O, LSE, dQ, dK, dV) out.  Inputs should be pinned
        for the copies to overlap; outputs (``out``: dict of pinned tensors) are filled in place.
        ``deterministic`` runs the backward pass through fa_bwd_deterministic; ``block_index``
        (a binding.BlockIndex with one mask shared by all heads) runs the block-sparse calls."""
        B, H, N, d = self.shape
        if block_index is not None and block_index.mask_heads != 1:
            raise ValueError("the host pipeline takes a block mask shared by every head")
        cur = torch.cuda.current_stream(self.device)
        if out is None:
            out = {name: torch.empty(self.shape, dtype=torch.bfloat16).pin_memory()
                   for name in ("O", "dQ", "dK", "dV")}
            out["LSE"] = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        for s in (self.s_in, self.s_comp, self.s_out):
            s.wait_stream(cur)
        if kv_lens is not None:
            with torch.cuda.stream(self.s_in):
                self.kv.copy_(kv_lens.to(torch.int32), non_blocking=True)
        for b0, b1, h0, h1 in self.plan:
            sl = (slice(b0, b1), slice(h0, h1))
            with torch.cuda.stream(self.s_in):
                for dst, src in ((self.q, q), (self.k, k), (self.v, v), (self.do, do)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(self.s_in)
            self.s_comp.wait_event(ev_in)
            with torch.cuda.stream(self.s_comp):
                view = lambda t: t[sl]  # noqa: E731  [b1-b0, h1-h0, N, d], contiguous
                kv = self.kv[b0:b1] if kv_lens is not None else None
                o, lse = view(self.o), self.lse[sl]
                qkv = (view(self.q), view(self.k), view(self.v))
                grads = dict(dq=view(self.dq), dk=view(self.dk), dv=view(self.dv),
                             workspace=self.workspace, stream=self.s_comp)
                if block_index is not None:
                    binding.fa_fwd_block_sparse(*qkv, block_index, causal=causal, scale=scale,
                                                kv_lens=kv, out=o, lse=lse, stream=self.s_comp)
                    binding.fa_bwd_block_sparse(*qkv, o, view(self.do), lse, block_index,
                                                causal=causal, scale=scale, kv_lens=kv,
                                                deterministic=deterministic, **grads)
                else:
                    binding.fa_fwd(*qkv, causal=causal, scale=scale, kv_lens=kv, out=o, lse=lse,
                                   stream=self.s_comp)
                    bwd = binding.fa_bwd_deterministic if deterministic else binding.fa_bwd
                    bwd(*qkv, o, view(self.do), lse, causal=causal, scale=scale, kv_lens=kv,
                        **grads)
                ev_comp = torch.cuda.Event()
                ev_comp.record(self.s_comp)
            self.s_out.wait_event(ev_comp)
            with torch.cuda.stream(self.s_out):
                for src, name in ((self.o, "O"), (self.dq, "dQ"), (self.dk, "dK"), (self.dv, "dV")):
                    out[name][sl].copy_(src[sl], non_blocking=True)
                out["LSE"][sl].copy_(self.lse[sl], non_blocking=True)
        for s in (self.s_in, self.s_comp, self.s_out):
            cur.wait_stream(s)
        return out

    def transfer_bytes(self, with_kv=False):
        """(host-to-device, device-to-host) bytes of one run()."""
        B, H, N, d = self.shape
        t = B * H * N * d * 2
        return 4 * t + (4 * B if with_kv else 0), 4 * t + 4 * B * H * N


def attention_fwd_bwd_host(q, k, v, do, causal=False, scale=None, kv_lens=None,
                           heads_per_chunk=None):
    """One-shot convenience wrapper around HostAttention (allocates device buffers each call)."""
    B, H, N, d = q.shape
    ha = HostAttention(B, H, N, d, heads_per_chunk=heads_per_chunk)
    return ha.run(q, k, v, do, causal=causal, scale=scale, kv_lens=kv_lens)
