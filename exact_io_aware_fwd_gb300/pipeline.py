"""Host-resident forward + backward with copies overlapped with compute.

``HostAttention`` (dense and grouped-query [B, H, N, d] tensors) and ``VarlenHostAttention``
(packed variable-length [total, H, d] tensors) serve data that lives in (pinned) host memory:
the work is split into chunks that attention never mixes (whole heads, whole key/value-head
groups, whole sequences), and for each chunk Q, K, V, dO are copied in on one stream, the
library's forward and backward calls run on a compute stream, and O, LSE, dQ, dK, dV are copied
out on a third, ordered by CUDA events.  While chunk c computes, chunk c+1 is copied in and
chunk c-1 copied out.  Chunks alternate between `compute_streams` compute streams (each with its
own backward workspace), so that the last, partly filled wave of one chunk's kernels overlaps
the next chunk's kernels instead of idling SMs.  Only orchestration happens here; the arithmetic
is the library's kernels.
"""

from __future__ import annotations

import torch

from . import binding


def _chunks(B, H, target=16, heads_per_chunk=None):
    """(b0, b1, h0, h1) pieces, each a contiguous slice q[b0:b1, h0:h1] of a [B, H, N, d] tensor:
    about `target` pieces of whole batches when B >= target, otherwise head ranges of one batch
    (`heads_per_chunk` overrides the head-range width).  With grouped-query attention the
    `H` here counts key/value heads, each standing for its whole group of query heads."""
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


def _seq_chunks(lengths, target=16):
    """(b0, b1) runs of whole sequences, contiguous in a packed [total, ...] tensor, with about
    equal attention work each (a sequence of length L costs L^2; a causal mask halves every
    sequence's cost alike, so it does not change the split).  At most `target` runs; a run never
    splits a sequence.  Each cut goes on the side of the sequence that crosses the next equal
    share where the running work lands closer to that share, so a dominant sequence ends up in
    a run of its own."""
    work = [int(n) * int(n) for n in lengths]
    B, total = len(work), sum(work)
    if B == 0:
        return []
    share = total / max(1, min(target, B))
    runs, b0, acc = [], 0, 0
    for b in range(B):
        boundary = share * (len(runs) + 1)
        if (total > 0 and len(runs) + 1 < target and b > b0 and acc + work[b] > boundary
                and boundary - acc < acc + work[b] - boundary):
            runs.append((b0, b))  # cut before b: closer to the share
            b0 = b
            boundary = share * (len(runs) + 1)
        acc += work[b]
        if total > 0 and len(runs) + 1 < target and b + 1 < B and acc >= boundary:
            runs.append((b0, b + 1))
            b0 = b + 1
    runs.append((b0, B))
    return runs


class _Pipeline:
    """Streams, per-stream workspaces and CUDA-graph capture shared by the host pipelines."""

    def __init__(self, device, n_chunks, compute_streams, copy_streams):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        dev = self.device
        ncomp = max(1, min(compute_streams, n_chunks))
        ncopy = max(1, min(copy_streams, n_chunks))
        self.s_ins = [torch.cuda.Stream(dev) for _ in range(ncopy)]
        self.s_comps = [torch.cuda.Stream(dev) for _ in range(ncomp)]
        self.s_outs = [torch.cuda.Stream(dev) for _ in range(ncopy)]
        self._graph = None      # captured run (graph=True) and the arguments it was captured for
        self._graph_key = None

    def _streams_for(self, c):
        return (self.s_ins[c % len(self.s_ins)], self.s_comps[c % len(self.s_comps)],
                self.s_outs[c % len(self.s_outs)], self.workspaces[c % len(self.s_comps)])

    def _run(self, key, issue, graph):
        """Run `issue()` (which enqueues one whole run) eagerly, or through a CUDA graph captured
        the first time `key` (buffer addresses and arguments) is seen and replayed afterwards."""
        if not graph:
            issue()
            return
        if self._graph is None or self._graph_key != key:
            issue()  # first use of these buffers: library set-up happens outside the capture
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            capture = torch.cuda.Stream(self.device)
            with torch.cuda.graph(g, stream=capture):
                issue()
            self._graph, self._graph_key = g, key
        self._graph.replay()

    def _fork(self):
        cur = torch.cuda.current_stream(self.device)
        streams = [*self.s_ins, *self.s_comps, *self.s_outs]
        for s in streams:
            s.wait_stream(cur)
        return cur, streams

    @staticmethod
    def _join(cur, streams):
        for s in streams:
            cur.wait_stream(s)


class HostAttention(_Pipeline):
    """Device buffers, streams and events for repeated host-to-host fwd + bwd of one shape:
    Q, dO, O, dQ [B, H, N, d]; K, V, dK, dV [B, Hkv, N, d] (Hkv = H unless grouped-query);
    LSE [B, H, N].  With Hkv < H a chunk holds whole key/value heads with their query heads."""

    # Defaults measured on GB300 (pinned host buffers, long-causal 1x32x16384x128): 16 chunks on 3
    # compute streams 6.90 ms per step, 8 chunks on 1 stream 7.74 ms; a second copy stream per
    # direction was slower (the host link, not one copy engine, bounds the copies).
    def __init__(self, B, H, N, d, device=None, heads_per_chunk=None, chunks=16,
                 compute_streams=3, copy_streams=1, Hkv=None):
        Hkv = H if Hkv is None else Hkv
        if Hkv <= 0 or H % Hkv != 0:
            raise ValueError("H must be a multiple of Hkv")
        self.shape, self.Hkv, self.group = (B, H, N, d), Hkv, H // Hkv
        G = self.group
        kv_per_chunk = None if heads_per_chunk is None else max(1, heads_per_chunk // G)
        # chunks in key/value-head units: (b0, b1, g0, g1) -> query heads [g0 G, g1 G)
        self.plan = list(_chunks(B, Hkv, target=chunks, heads_per_chunk=kv_per_chunk))
        super().__init__(device, len(self.plan), compute_streams, copy_streams)
        dev = self.device
        q_shape, kv_shape = (B, H, N, d), (B, Hkv, N, d)
        mk = lambda shape: torch.empty(shape, dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.q, self.do, self.o, self.dq = (mk(q_shape) for _ in range(4))
        self.k, self.v, self.dk, self.dv = (mk(kv_shape) for _ in range(4))
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.kv = torch.empty((B,), dtype=torch.int32, device=dev)
        self.kv_host = torch.zeros((B,), dtype=torch.int32).pin_memory()  # staging for kv_lens
        self._kv_last = None
        max_heads = max((b1 - b0) * (g1 - g0) * G for b0, b1, g0, g1 in self.plan)
        # chunks on one compute stream run one after another, so one workspace per stream
        self.workspaces = [torch.empty(binding.fa_bwd_workspace_size(1, max_heads, N, d),
                                       dtype=torch.uint8, device=dev) for _ in self.s_comps]

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
        if block_index is not None and (block_index.mask_heads != 1 or self.group != 1):
            raise ValueError("the host pipeline takes a block mask shared by every head, "
                             "without grouped-query attention")
        if out is None:
            q_shape, kv_shape = (B, H, N, d), (B, self.Hkv, N, d)
            out = {name: torch.empty(shape, dtype=torch.bfloat16).pin_memory()
                   for name, shape in (("O", q_shape), ("dQ", q_shape), ("dK", kv_shape),
                                       ("dV", kv_shape))}
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
        key = (tuple(t.data_ptr() for t in (q, k, v, do)), tuple(sorted(
            (n, t.data_ptr()) for n, t in out.items())), causal, scale, has_kv, deterministic,
            id(block_index))
        self._run(key, lambda: self._issue(*args), graph)
        return out

    def _issue(self, q, k, v, do, causal, scale, has_kv, out, deterministic, block_index):
        """Enqueue one run on the pipeline's streams, ordered after the current stream."""
        G = self.group
        cur, streams = self._fork()
        ev_kv = None
        if has_kv:
            with torch.cuda.stream(self.s_ins[0]):
                self.kv.copy_(self.kv_host, non_blocking=True)
                ev_kv = torch.cuda.Event()
                ev_kv.record(self.s_ins[0])
        for c, (b0, b1, g0, g1) in enumerate(self.plan):
            slq = (slice(b0, b1), slice(g0 * G, g1 * G))  # query heads of the chunk
            slk = (slice(b0, b1), slice(g0, g1))          # its key/value heads
            s_in, s_comp, s_out, workspace = self._streams_for(c)
            with torch.cuda.stream(s_in):
                for dst, src, sl in ((self.q, q, slq), (self.k, k, slk), (self.v, v, slk),
                                     (self.do, do, slq)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            if ev_kv is not None:
                s_comp.wait_event(ev_kv)
            with torch.cuda.stream(s_comp):
                kv = self.kv[b0:b1] if has_kv else None
                o, lse, dov = self.o[slq], self.lse[slq], self.do[slq]
                qkv = (self.q[slq], self.k[slk], self.v[slk])
                grads = dict(dq=self.dq[slq], dk=self.dk[slk], dv=self.dv[slk],
                             workspace=workspace, stream=s_comp)
                if block_index is not None:
                    binding.fa_fwd_block_sparse(*qkv, block_index, causal=causal, scale=scale,
                                                kv_lens=kv, out=o, lse=lse, stream=s_comp)
                    binding.fa_bwd_block_sparse(*qkv, o, dov, lse, block_index,
                                                causal=causal, scale=scale, kv_lens=kv,
                                                deterministic=deterministic, **grads)
                elif G > 1:
                    binding.fa_fwd_gqa(*qkv, causal=causal, scale=scale, kv_lens=kv, out=o,
                                       lse=lse, stream=s_comp)
                    binding.fa_bwd_gqa(*qkv, o, dov, lse, causal=causal, scale=scale,
                                       kv_lens=kv, deterministic=deterministic, **grads)
                else:
                    binding.fa_fwd(*qkv, causal=causal, scale=scale, kv_lens=kv, out=o, lse=lse,
                                   stream=s_comp)
                    bwd = binding.fa_bwd_deterministic if deterministic else binding.fa_bwd
                    bwd(*qkv, o, dov, lse, causal=causal, scale=scale, kv_lens=kv, **grads)
                ev_comp = torch.cuda.Event()
                ev_comp.record(s_comp)
            s_out.wait_event(ev_comp)
            with torch.cuda.stream(s_out):
                for src, name, sl in ((self.o, "O", slq), (self.dq, "dQ", slq),
                                      (self.dk, "dK", slk), (self.dv, "dV", slk),
                                      (self.lse, "LSE", slq)):
                    out[name][sl].copy_(src[sl], non_blocking=True)
        self._join(cur, streams)

    def transfer_bytes(self, with_kv=False):
        """(host-to-device, device-to-host) bytes of one run()."""
        B, H, N, d = self.shape
        tq, tkv = B * H * N * d * 2, B * self.Hkv * N * d * 2
        return 2 * tq + 2 * tkv + (4 * B if with_kv else 0), 2 * tq + 2 * tkv + 4 * B * H * N


class VarlenHostAttention(_Pipeline):
    """The same for a packed variable-length batch: Q, dO, O, dQ [total, H, d]; K, V, dK, dV
    [total, Hkv, d]; LSE [H, total]; sequence b holds tokens [cu_seqlens[b], cu_seqlens[b+1]).
    A chunk is a run of whole sequences (a contiguous token range) with about equal work; its
    cu_seqlens, rebased to the run's first token, are uploaded once here."""

    def __init__(self, cu_seqlens, H, d, device=None, chunks=16, compute_streams=3,
                 copy_streams=1, Hkv=None):
        cu = [int(x) for x in torch.as_tensor(cu_seqlens).tolist()]
        if len(cu) < 2 or cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
            raise ValueError("cu_seqlens must start at 0 and not decrease")
        Hkv = H if Hkv is None else Hkv
        if Hkv <= 0 or H % Hkv != 0:
            raise ValueError("H must be a multiple of Hkv")
        self.cu, self.H, self.Hkv, self.d = cu, H, Hkv, d
        self.total = total = cu[-1]
        lengths = [b - a for a, b in zip(cu, cu[1:])]
        # runs with no token have nothing to copy or compute
        self.plan = [(b0, b1) for b0, b1 in _seq_chunks(lengths, target=chunks) if cu[b1] > cu[b0]]
        super().__init__(device, max(1, len(self.plan)), compute_streams, copy_streams)
        dev = self.device
        mk = lambda heads: torch.empty((total, heads, d), dtype=torch.bfloat16, device=dev)  # noqa: E731
        self.q, self.do, self.o, self.dq = (mk(H) for _ in range(4))
        self.k, self.v, self.dk, self.dv = (mk(Hkv) for _ in range(4))
        # LSE of chunk c as its own [H, tokens] block at H * (first token): the kernels write a
        # call's LSE as [H, total of the call]
        self.lse = torch.empty((H * total,), dtype=torch.float32, device=dev)
        self.cus = [torch.tensor([x - cu[b0] for x in cu[b0:b1 + 1]], dtype=torch.int32,
                                 device=dev) for b0, b1 in self.plan]
        self.max_len = [max(lengths[b0:b1]) for b0, b1 in self.plan]
        need = max((binding.fa_bwd_varlen_workspace_size(b1 - b0, cu[b1] - cu[b0], H, d)
                    for b0, b1 in self.plan), default=256)
        self.workspaces = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in self.s_comps]

    def run(self, q, k, v, do, causal=False, scale=None, out=None, deterministic=False,
            graph=False):
        """Host tensors in -> host tensors (O, LSE, dQ, dK, dV) out, as HostAttention.run."""
        H, Hkv, d, total = self.H, self.Hkv, self.d, self.total
        if out is None:
            out = {name: torch.empty((total, heads, d), dtype=torch.bfloat16).pin_memory()
                   for name, heads in (("O", H), ("dQ", H), ("dK", Hkv), ("dV", Hkv))}
            out["LSE"] = torch.empty((H, total), dtype=torch.float32).pin_memory()
        key = (tuple(t.data_ptr() for t in (q, k, v, do)), tuple(sorted(
            (n, t.data_ptr()) for n, t in out.items())), causal, scale, deterministic)
        self._run(key, lambda: self._issue(q, k, v, do, causal, scale, out, deterministic), graph)
        return out

    def _issue(self, q, k, v, do, causal, scale, out, deterministic):
        H = self.H
        cur, streams = self._fork()
        for c, (b0, b1) in enumerate(self.plan):
            t0, t1 = self.cu[b0], self.cu[b1]
            sl = slice(t0, t1)
            s_in, s_comp, s_out, workspace = self._streams_for(c)
            with torch.cuda.stream(s_in):
                for dst, src in ((self.q, q), (self.k, k), (self.v, v), (self.do, do)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            lse = self.lse[H * t0:H * t1].view(H, t1 - t0)
            with torch.cuda.stream(s_comp):
                qkv = (self.q[sl], self.k[sl], self.v[sl])
                binding.fa_fwd_varlen(*qkv, self.cus[c], self.max_len[c], causal=causal,
                                      scale=scale, out=self.o[sl], lse=lse, stream=s_comp)
                binding.fa_bwd_varlen(*qkv, self.o[sl], self.do[sl], lse, self.cus[c],
                                      self.max_len[c], causal=causal, scale=scale,
                                      deterministic=deterministic, dq=self.dq[sl], dk=self.dk[sl],
                                      dv=self.dv[sl], workspace=workspace, stream=s_comp)
                ev_comp = torch.cuda.Event()
                ev_comp.record(s_comp)
            s_out.wait_event(ev_comp)
            with torch.cuda.stream(s_out):
                for src, name in ((self.o, "O"), (self.dq, "dQ"), (self.dk, "dK"),
                                  (self.dv, "dV")):
                    out[name][sl].copy_(src[sl], non_blocking=True)
                for h in range(H):  # one contiguous row of LSE per head
                    out["LSE"][h, sl].copy_(lse[h], non_blocking=True)
        self._join(cur, streams)

    def transfer_bytes(self):
        """(host-to-device, device-to-host) bytes of one run()."""
        tq, tkv = self.total * self.H * self.d * 2, self.total * self.Hkv * self.d * 2
        return 2 * tq + 2 * tkv, 2 * tq + 2 * tkv + 4 * self.H * self.total


def attention_fwd_bwd_host(q, k, v, do, causal=False, scale=None, kv_lens=None,
                           heads_per_chunk=None, chunks=16, compute_streams=3, copy_streams=1):
    """One-shot convenience wrapper around HostAttention (allocates device buffers each call);
    K and V may have fewer heads than Q (grouped-query)."""
    B, H, N, d = q.shape
    ha = HostAttention(B, H, N, d, heads_per_chunk=heads_per_chunk, chunks=chunks,
                       compute_streams=compute_streams, copy_streams=copy_streams,
                       Hkv=k.shape[1])
    return ha.run(q, k, v, do, causal=causal, scale=scale, kv_lens=kv_lens)
