"""Host-resident forward + backward with copies overlapped with compute.

``attention_fwd_bwd_host`` is the call for data that lives in (pinned) host memory: it splits the
work into chunks of whole heads, and for each chunk copies Q, K, V, dO in on one stream, runs
fa_fwd and fa_bwd on a compute stream and copies O, LSE, dQ, dK, dV out on a third, with CUDA
events ordering them.  Chunks are independent (attention never mixes heads), so while chunk c
computes, chunk c+1 is copied in and chunk c-1 copied out.  Chunks alternate between
`compute_streams` compute streams (each with its own workspace), so that the last, partly
filled wave of one chunk's kernels overlaps the next chunk's kernels instead of idling SMs.
Only orchestration happens here; the arithmetic is the library's kernels.
"""

from __future__ import annotations

import torch

from . import binding


def _chunks(B, H, target=16, heads_per_chunk=None):
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

    # Defaults measured on GB300 (pinned host buffers, long-causal 1x32x16384x128): 16 chunks on 3
    # compute streams 6.90 ms per step, 8 chunks on 1 stream 7.74 ms; a second copy stream per
    # direction was slower (the host link, not one copy engine, bounds the copies).
    def __init__(self, B, H, N, d, device=None, heads_per_chunk=None, chunks=16,
                 compute_streams=3, copy_streams=1):
        self.shape = (B, H, N, d)
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        dev = self.device
        mk = lambda: torch.empty(self.shape, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.q, self.k, self.v, self.do = mk(), mk(), mk(), mk()
        self.o, self.dq, self.dk, self.dv = mk(), mk(), mk(), mk()
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.kv = torch.empty((B,), dtype=torch.int32, device=dev)
        self.kv_host = torch.zeros((B,), dtype=torch.int32).pin_memory()  # staging for kv_lens
        self._kv_last = None
        self._graph = None      # captured run (graph=True) and the arguments it was captured for
        self._graph_key = None
        self.plan = list(_chunks(B, H, target=chunks, heads_per_chunk=heads_per_chunk))
        max_heads = max((b1 - b0) * (h1 - h0) for b0, b1, h0, h1 in self.plan)
        ncomp = max(1, min(compute_streams, len(self.plan)))
        # chunks on one compute stream run one after another, so one workspace per stream
        self.workspaces = [torch.empty(binding.fa_bwd_workspace_size(1, max_heads, N, d),
                                       dtype=torch.uint8, device=dev) for _ in range(ncomp)]
        ncopy = max(1, min(copy_streams, len(self.plan)))
        self.s_ins = [torch.cuda.Stream(dev) for _ in range(ncopy)]
        self.s_comps = [torch.cuda.Stream(dev) for _ in range(ncomp)]
        self.s_outs = [torch.cuda.Stream(dev) for _ in range(ncopy)]

    def run(self, q, k, v, do, causal=False, scale=None, kv_lens=None, out=None,
            deterministic=False, block_index=None, graph=False):
        """Host tensors in -> host tensors (O, LSE, dQ, dK, dV) out.  Inputs should be pinned
        for the copies to overlap; outputs (``out``: dict of pinned tensors) are filled in place.
        ``deterministic`` runs the backward pass through fa_bwd_deterministic; ``block_index``
        (a binding.BlockIndex with one mask shared by all heads) runs the block-sparse calls.

        ``graph=True`` captures the whole run (copies, kernels, cross-stream events) in a CUDA
        graph the first time it sees these buffers and arguments, and replays it afterwards:
        one launch instead of hundreds of host calls per run, which matters when the chunks are
        short.  Replays read the inputs' current contents; new buffers or arguments recapture."""
        B, H, N, d = self.shape
        if block_index is not None and block_index.mask_heads != 1:
            raise ValueError("the host pipeline takes a block mask shared by every head")
        if out is None:
            out = {name: torch.empty(self.shape, dtype=torch.bfloat16).pin_memory()
                   for name in ("O", "dQ", "dK", "dV")}
            out["LSE"] = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        has_kv = kv_lens is not None
        if has_kv:
            vals = torch.as_tensor(kv_lens).to(dtype=torch.int32, device="cpu")
            if self._kv_last is None or not torch.equal(vals, self._kv_last):
                # the staging buffer may still be read by a run in flight
                torch.cuda.synchronize(self.device)
                self.kv_host.copy_(vals)
                self._kv_last = vals.clone()
        args = (q, k, v, do, causal, scale, has_kv, out, deterministic, block_index)
        if not graph:
            self._issue(*args)
            return out
        key = (tuple(t.data_ptr() for t in (q, k, v, do)), tuple(sorted(
            (n, t.data_ptr()) for n, t in out.items())), causal, scale, has_kv, deterministic,
            id(block_index))
        if self._graph is None or self._graph_key != key:
            self._issue(*args)  # first use of these buffers: library set-up happens outside
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            capture = torch.cuda.Stream(self.device)
            with torch.cuda.graph(g, stream=capture):
                self._issue(*args)
            self._graph, self._graph_key = g, key
        self._graph.replay()
        return out

    def _issue(self, q, k, v, do, causal, scale, has_kv, out, deterministic, block_index):
        """Enqueue one run on the pipeline's streams, ordered after the current stream."""
        cur = torch.cuda.current_stream(self.device)
        streams = [*self.s_ins, *self.s_comps, *self.s_outs]
        for s in streams:
            s.wait_stream(cur)
        ev_kv = None
        if has_kv:
            with torch.cuda.stream(self.s_ins[0]):
                self.kv.copy_(self.kv_host, non_blocking=True)
                ev_kv = torch.cuda.Event()
                ev_kv.record(self.s_ins[0])
        for c, (b0, b1, h0, h1) in enumerate(self.plan):
            sl = (slice(b0, b1), slice(h0, h1))
            s_comp = self.s_comps[c % len(self.s_comps)]
            workspace = self.workspaces[c % len(self.s_comps)]
            s_in = self.s_ins[c % len(self.s_ins)]
            s_out = self.s_outs[c % len(self.s_outs)]
            with torch.cuda.stream(s_in):
                for dst, src in ((self.q, q), (self.k, k), (self.v, v), (self.do, do)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            if ev_kv is not None:
                s_comp.wait_event(ev_kv)
            with torch.cuda.stream(s_comp):
                view = lambda t: t[sl]  # noqa: E731  [b1-b0, h1-h0, N, d], contiguous
                kv = self.kv[b0:b1] if has_kv else None
                o, lse = view(self.o), self.lse[sl]
                qkv = (view(self.q), view(self.k), view(self.v))
                grads = dict(dq=view(self.dq), dk=view(self.dk), dv=view(self.dv),
                             workspace=workspace, stream=s_comp)
                if block_index is not None:
                    binding.fa_fwd_block_sparse(*qkv, block_index, causal=causal, scale=scale,
                                                kv_lens=kv, out=o, lse=lse, stream=s_comp)
                    binding.fa_bwd_block_sparse(*qkv, o, view(self.do), lse, block_index,
                                                causal=causal, scale=scale, kv_lens=kv,
                                                deterministic=deterministic, **grads)
                else:
                    binding.fa_fwd(*qkv, causal=causal, scale=scale, kv_lens=kv, out=o, lse=lse,
                                   stream=s_comp)
                    bwd = binding.fa_bwd_deterministic if deterministic else binding.fa_bwd
                    bwd(*qkv, o, view(self.do), lse, causal=causal, scale=scale, kv_lens=kv,
                        **grads)
                ev_comp = torch.cuda.Event()
                ev_comp.record(s_comp)
            s_out.wait_event(ev_comp)
            with torch.cuda.stream(s_out):
                for src, name in ((self.o, "O"), (self.dq, "dQ"), (self.dk, "dK"), (self.dv, "dV")):
                    out[name][sl].copy_(src[sl], non_blocking=True)
                out["LSE"][sl].copy_(self.lse[sl], non_blocking=True)
        for s in streams:
            cur.wait_stream(s)

    def transfer_bytes(self, with_kv=False):
        """(host-to-device, device-to-host) bytes of one run()."""
        B, H, N, d = self.shape
        t = B * H * N * d * 2
        return 4 * t + (4 * B if with_kv else 0), 4 * t + 4 * B * H * N


def attention_fwd_bwd_host(q, k, v, do, causal=False, scale=None, kv_lens=None,
                           heads_per_chunk=None, chunks=16, compute_streams=3, copy_streams=1):
    """One-shot convenience wrapper around HostAttention (allocates device buffers each call)."""
    B, H, N, d = q.shape
    ha = HostAttention(B, H, N, d, heads_per_chunk=heads_per_chunk, chunks=chunks,
                       compute_streams=compute_streams, copy_streams=copy_streams)
    return ha.run(q, k, v, do, causal=causal, scale=scale, kv_lens=kv_lens)
