"""Benchmark of the exact-attention hot path (forward + backward) on one GB300.

A step is one pass of the whole path over one batch: fa_fwd, then fa_bwd's three stages
(preprocess, dK/dV with dQ accumulation, dQ convert).  The metric is attention TFLOPS with the
pages' convention (4 N^2 d forward + 10 N^2 d backward per head, halved when causal).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the long-context causal case (B=1, H=32, N=16384, d=128), whose inputs
(4 x 134 MB) are larger than the 129 MB L2, so no flush is needed between steps; workloads
whose inputs fit in L2 get a 256 MB write between steps, outside the per-step events.
With torchrun (N > 1) every rank runs an independent replica (the path does not shard across
GPUs); the timed region is bracketed by barriers and the max over ranks is reported.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_io_aware_fwd_gb300.workloads import (BY_NAME, HEADLINE, workload_block_mask,  # noqa: E402
                                                 workload_inputs)

METRIC = "attention fwd/bwd TFLOPS (bf16, 1\u00d7GB300) and % of dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Sources whose change invalidates a recorded DRAM-traffic figure, per kernel (the launch setup
# in fa_api.cu and the shared headers count for every kernel).
_COMMON = ["exact_io_aware_fwd_gb300/csrc/fa_api.cu", "exact_io_aware_fwd_gb300/csrc/fa_internal.h",
           "exact_io_aware_fwd_gb300/csrc/sm103.cuh"]
SOURCES_FOR_TRAFFIC = {
    "fwd": _COMMON + ["exact_io_aware_fwd_gb300/csrc/fa_fwd.cu"],
    "bwd": _COMMON + ["exact_io_aware_fwd_gb300/csrc/fa_bwd.cu",
                      "exact_io_aware_fwd_gb300/csrc/fa_bwd_dq.cu"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE.name, choices=sorted(BY_NAME))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--bwd", default="atomic", choices=["atomic", "deterministic"],
                    help="backward entry: fa_bwd (dQ by fp32 atomics) or fa_bwd_deterministic")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ingest-ncu", metavar="CSV", default=None,
                    help="record the DRAM bytes of an ncu launch list of --workload in "
                         "profiles/traffic.json and exit (no GPU needed)")
    ap.add_argument("--ncu-command", default="", help="the ncu command that wrote --ingest-ncu")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=None,
                    help="override H (smaller profiling captures of the same shape); the line "
                         "is then not the headline measurement")
    return ap.parse_args()


# ------------------------------------------------------------------------------- distributed
def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def sources_digest(kind):
    """Short hash of the kernel sources of `kind` ("fwd" or "bwd")."""
    h = hashlib.sha256()
    for rel in SOURCES_FOR_TRAFFIC[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch (per call, for a multi-kernel backward call) from the committed ncu
    summary, if it was taken on the current sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if kernel.startswith("fa_bwd"):  # a backward call of several kernels: their sum per call
        kernel = "bwd_step"
    e = d.get(f"{kernel}@{workload}")
    kind = "fwd" if kernel.startswith("fwd") else "bwd"
    if not e or e.get("sources") != sources_digest(kind):
        return None
    return e.get("dram_bytes_per_launch")


def ingest_ncu(csv_path, workload, command):
    """Record the DRAM bytes of an ncu launch list (``--metrics gpu__time_duration.sum,
    dram__bytes_read.sum,dram__bytes_write.sum --csv``) of `workload` in profiles/traffic.json:
    per kernel the mean per launch, and "bwd_step" = the sum of the backward kernels' means."""
    import collections
    import csv
    import re

    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr = rows[hi]
    col = {k: hdr.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit",
                                     "Metric Value")}
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1, "usecond": 1e3,
             "msecond": 1e6, "ns": 1, "us": 1e3, "ms": 1e6}
    launches = collections.defaultdict(dict)
    names = {}
    for r in rows[hi + 1:]:
        v = float(r[col["Metric Value"]].replace(",", "")) * scale.get(r[col["Metric Unit"]], 1)
        launches[r[col["ID"]]][r[col["Metric Name"]]] = v
        names[r[col["ID"]]] = r[col["Kernel Name"]]
    agg = collections.defaultdict(list)
    for i, m in launches.items():
        base = re.search(r"(\w+_kernel)", names[i]).group(1)
        agg[base].append(m)
    p = os.path.join(ROOT, "profiles", "traffic.json")
    d = json.load(open(p)) if os.path.exists(p) else {}
    d["_note"] = ("DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, mean over "
                  "the launches of the list) from full-size launch lists; 'command' is the ncu "
                  "command, 'sources' the digest of the kernel's sources it ran; bench.py reports "
                  "a figure only while the digest matches")
    step = {"dram_bytes_per_launch": 0.0, "read": 0.0, "write": 0.0, "ns_per_launch": 0.0}
    for base, ms in agg.items():
        mean = lambda k: sum(m[k] for m in ms) / len(ms)  # noqa: E731
        e = {"dram_bytes_per_launch": mean("dram__bytes_read.sum") + mean("dram__bytes_write.sum"),
             "read": mean("dram__bytes_read.sum"), "write": mean("dram__bytes_write.sum"),
             "ns_per_launch": mean("gpu__time_duration.sum"), "launches": len(ms),
             "sources": sources_digest("fwd" if base.startswith("fwd") else "bwd"),
             "command": command}
        d[f"{base}@{workload}"] = e
        if base.startswith("bwd_"):
            for k in step:
                step[k] += e[k]
    if step["ns_per_launch"] > 0:
        d[f"bwd_step@{workload}"] = dict(step, sources=sources_digest("bwd"), command=command)
    with open(p, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")


class _Nvml:
    """The few read-only NVML queries the clock sampler needs, through ctypes on the driver's
    libnvidia-ml (no Python package needed).  None of these calls changes any GPU setting."""

    CLOCK_SM = 1
    # clock event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x40: "sw_thermal_slowdown",
               0x80: "hw_thermal_slowdown", 0x100: "hw_power_brake_slowdown"}

    def __init__(self, index):
        import ctypes

        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML device")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        v = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) != 0:
            raise OSError("no max clock")
        self.max_sm = v.value

    def sample(self):
        v, r = self.c.c_uint(), self.c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.c.byref(v)) != 0:
            return None
        if self.reasons_fn(self.h, self.c.byref(r)) != 0:
            return None
        return v.value, r.value


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: every 10 ms through NVML
    (samples outside [mark_start, mark_end] are dropped), else every 200 ms through nvidia-smi
    (all samples kept)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []       # nvidia-smi rows
        self.samples = []    # NVML (time, sm_mhz, reason bits)
        self.window = None
        self._stop = threading.Event()
        self._proc = None
        self._thread = None
        try:
            self._nvml = _Nvml(gpu_index)
        except (OSError, AttributeError):
            self._nvml = None

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self._proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _poll(self):
        while not self._stop.is_set():
            got = self._nvml.sample()
            if got is not None:
                self.samples.append((time.perf_counter(), *got))
            time.sleep(0.01)

    def _read(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def mark(self, t_start, t_end):
        """The host-clock interval of the timed region (first launch .. final synchronize)."""
        self.window = (t_start, t_end)

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        if self._nvml is not None:
            lo, hi = self.window if self.window else (float("-inf"), float("inf"))
            inside = [(mhz, bits) for t, mhz, bits in self.samples if lo <= t <= hi]
            if not inside:
                return {"sm_mhz": None, "sm_max_mhz": self._nvml.max_sm, "reasons": ["unsampled"],
                        "samples": 0, "source": "nvml"}
            reasons = sorted({name for _, bits in inside for bit, name in _Nvml.REASONS.items()
                              if bits & bit})
            return {"sm_mhz": statistics.median(m for m, _ in inside),
                    "sm_max_mhz": self._nvml.max_sm, "reasons": reasons,
                    "samples": len(inside), "source": "nvml, every 10 ms"}
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(self.rows), "source": "nvidia-smi, every 200 ms"}


# ------------------------------------------------------------------------------- oracle timing
def oracle_row_block(q, k, v, do, causal, scale, kv_len, rows, block_mask=None):
    """One bounded sample of the oracle: forward + backward restricted to a block of query rows
    (O, LSE, D, dQ of those rows and their contributions to dK, dV).  Returns the credited
    FLOPs with the metric's convention: 14 d per visible (query, key) pair."""
    import oracle

    st = oracle.row_statistics(q, k, v, do, scale, causal, kv_len, rows, block_mask)
    oracle.key_gradients(q, k, v, do, scale, st["LSE"], st["D"], causal, kv_len, rows=rows,
                         block_mask=block_mask)
    n = k.shape[0]
    lim = n if kv_len is None else int(kv_len)
    if block_mask is not None:
        keys = np.arange(n)
        vis = block_mask[(rows // 128)[:, None], (keys // 128)[None, :]] != 0
        vis &= keys[None, :] < lim
        if causal:
            vis &= keys[None, :] <= rows[:, None]
        return 14.0 * q.shape[1] * float(vis.sum())
    visible = np.minimum(rows + 1, lim) if causal else np.full(len(rows), lim)
    return 14.0 * q.shape[1] * float(visible.sum())


def cpu_sample_inputs(w, q, k, v, do, kv, i=0):
    """The i-th (batch, head) slice in order, head 0 first (variable-length: the i-th sequence's
    head 0; kv is then cu_seqlens): (q, k, v, do, kv_len, n, label) as fp64 arrays plus the key
    length, the row count and a label; None past the last slice."""
    if w.seqlen_range is not None:
        if i >= w.B:
            return None
        s0, s1 = int(kv[i]), int(kv[i + 1])
        f = lambda t: t[s0:s1, 0].float().numpy().astype(np.float64)  # noqa: E731
        return f(q), f(k), f(v), f(do), None, s1 - s0, f"sequence {i} head 0"
    if i >= w.B * w.H:
        return None
    b, h = divmod(i, w.H)
    hk = h // (w.H // w.kv_heads)
    fq = lambda t: t[b, h].float().numpy().astype(np.float64)  # noqa: E731
    fk = lambda t: t[b, hk].float().numpy().astype(np.float64)  # noqa: E731
    kv_len = int(kv[b]) if kv is not None else None
    return fq(q), fk(k), fk(v), fq(do), kv_len, w.N, f"(b,h)=({b},{h})"


def time_oracle_once(w, q, k, v, do, kv, min_seconds=0.0, block=2048):
    """The oracle on blocks of `block` query rows, from a head's last rows backwards (the most
    keys under a causal mask) and head after head, until at least `min_seconds` have passed (one
    block when 0).  Returns (credited FLOPs, seconds, description of the sample)."""
    mask = workload_block_mask(w)
    mask = None if mask is None else mask.numpy()
    flops, dt, parts = 0.0, 0.0, []
    i = 0
    while True:
        sl = cpu_sample_inputs(w, q, k, v, do, kv, i)
        if sl is None:
            break
        qs, ks, vs, dos, kv_len, n, label = sl
        lo = n
        while lo > 0 and (dt < min_seconds or not parts and lo == n):
            rows = np.arange(max(0, lo - block), lo)
            t0 = time.perf_counter()
            flops += oracle_row_block(qs, ks, vs, dos, w.causal, w.scale, kv_len, rows, mask)
            dt += time.perf_counter() - t0
            lo = rows[0]
        parts.append(f"{label} query rows {lo}..{n - 1} of {n}")
        if dt >= min_seconds:
            break
        i += 1
    desc = "; ".join(parts) + ": O, LSE, dQ and their dK, dV contributions"
    return flops, dt, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def host_link_gbs(h_in, h_out, stream, reps=3):
    """Plain copy rates of the host link just before the end-to-end run: `h_in` (pinned) to a
    device buffer and back into `h_out` (pinned, same size), one direction at a time, then both
    at once on two streams ("both": bytes of both directions per second).  A slow end-to-end
    figure with normal rates here is the pipeline's; with low rates, the link's."""
    dbuf = torch.empty(h_in.shape, dtype=h_in.dtype, device=stream.device)
    dbuf2 = torch.empty(h_in.shape, dtype=h_in.dtype, device=stream.device)
    nbytes = h_in.numel() * h_in.element_size()
    rates = {}
    for name, copy in (("h2d", lambda: dbuf.copy_(h_in, non_blocking=True)),
                       ("d2h", lambda: h_out.copy_(dbuf, non_blocking=True))):
        copy()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            copy()
        b.record(stream)
        b.synchronize()
        rates[name] = reps * nbytes / (a.elapsed_time(b) * 1e6)
    other = torch.cuda.Stream(stream.device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    other.wait_stream(stream)
    for _ in range(reps):
        dbuf2.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(other):
            h_out.copy_(dbuf, non_blocking=True)
    stream.wait_stream(other)
    b.record(stream)
    b.synchronize()
    rates["both"] = 2 * reps * nbytes / (a.elapsed_time(b) * 1e6)
    del dbuf, dbuf2
    return rates


# ------------------------------------------------------------------------------- arms
def workload_config(w, extra, args, world):
    """The line's `config`: the workload's name and shape; `extra` is kv_lens (dense, may be
    None) or cu_seqlens (variable-length).  Both arms print the same object for the same
    arguments; how each arm treats L2 is a key of its own beside it."""
    varlen = w.seqlen_range is not None
    kv = None if varlen else extra
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "kv_lens": None if kv is None else kv.tolist(),
            "parallelism": f"replicas x{world}", "bwd": args.bwd, "block_mask": w.block_mask,
            "Hkv": w.kv_heads, "seqlens": extra.diff().tolist() if varlen else None}


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    q, k, v, do, kv = workload_inputs(w)
    times, flops = [], 0.0
    sample = ""
    for step in range(args.warmup + args.steps):
        f, dt, sample = time_oracle_once(w, q, k, v, do, kv)
        if step >= args.warmup:
            times.append(dt)
            flops = f
    total = sum(times)
    value = flops * len(times) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, kv, args, world),
        "l2": "n/a (CPU oracle)",
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample,
                         "full_step_seconds_extrapolated": sum(w.flops()) / (value * 1e12)},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, world, rank, local):
    import exact_io_aware_fwd_gb300 as fa

    fa.build()
    fa.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    varlen = w.seqlen_range is not None
    q, k, v, do, extra = workload_inputs(w)  # extra: kv_lens, or cu_seqlens when varlen
    kv = None if varlen else extra
    B, H, N, d = w.B, w.H, w.N, w.d
    stream = torch.cuda.current_stream()
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    kvd = kv.to(dev) if kv is not None else None
    cud = extra.to(dev) if varlen else None
    o = torch.empty_like(qd)
    lse_shape = (H, q.shape[0]) if varlen else (B, H, N)
    lse = torch.empty(lse_shape, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    if varlen:
        ws = torch.empty(fa.fa_bwd_varlen_workspace_size(B, q.shape[0], H, d), dtype=torch.uint8,
                         device=dev)
    else:
        ws = fa.workspace_for(qd)
    f_fwd, f_bwd = w.flops()

    det = args.bwd == "deterministic"
    mask = workload_block_mask(w)
    index = fa.fa_block_index_build(mask.to(dev), N) if mask is not None else None
    gqa = w.Hkv is not None and not varlen
    two_stage = det or index is not None or varlen or gqa
    stages = ["fwd", "bwd"] if two_stage else ["fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq_convert"]

    def step_two(evs=None):  # the forward call, then one backward call
        if evs is not None:
            evs[0].record(stream)
        if varlen:
            fa.fa_fwd_varlen(qd, kd, vd, cud, N, causal=w.causal, scale=w.scale, out=o, lse=lse)
            if evs is not None:
                evs[1].record(stream)
            fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, cud, N, causal=w.causal, scale=w.scale,
                             deterministic=det, dq=dq, dk=dk, dv=dv, workspace=ws)
        elif gqa:
            fa.fa_fwd_gqa(qd, kd, vd, causal=w.causal, scale=w.scale, out=o, lse=lse)
            if evs is not None:
                evs[1].record(stream)
            fa.fa_bwd_gqa(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale,
                          deterministic=det, dq=dq, dk=dk, dv=dv, workspace=ws)
        if varlen or gqa:
            if evs is not None:
                evs[2].record(stream)
            return
        if index is not None:
            fa.fa_fwd_block_sparse(qd, kd, vd, index, causal=w.causal, scale=w.scale,
                                   kv_lens=kvd, out=o, lse=lse)
        else:
            fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, kv_lens=kvd, out=o, lse=lse)
        if evs is not None:
            evs[1].record(stream)
        if index is not None:
            fa.fa_bwd_block_sparse(qd, kd, vd, o, dod, lse, index, causal=w.causal,
                                   scale=w.scale, kv_lens=kvd, deterministic=det, dq=dq, dk=dk,
                                   dv=dv, workspace=ws)
        else:
            fa.fa_bwd_deterministic(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale,
                                    kv_lens=kvd, dq=dq, dk=dk, dv=dv, workspace=ws)
        if evs is not None:
            evs[2].record(stream)

    def step(evs=None):
        if two_stage:
            return step_two(evs)
        if evs is not None:
            evs[0].record(stream)
        fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, kv_lens=kvd, out=o, lse=lse)
        if evs is not None:
            evs[1].record(stream)
        fa.fa_bwd_preprocess(o, dod, lse, ws)
        if evs is not None:
            evs[2].record(stream)
        fa.fa_bwd_dkdv(qd, kd, vd, dod, dk, dv, ws, causal=w.causal, scale=w.scale, kv_lens=kvd)
        if evs is not None:
            evs[3].record(stream)
        fa.fa_bwd_dq_convert(dq, ws, scale=w.scale)
        if evs is not None:
            evs[4].record(stream)

    for _ in range(args.warmup):
        step()
    st = fa.fa_get_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {fa.fa_status_string(st)}")

    # ---- device-timed region (inputs resident in HBM).  Inputs that fit in L2 would
    # stay there from one step to the next: then a 256 MB buffer is written between steps and
    # the step time is the sum of the per-step event intervals, which exclude those writes.
    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20
    in_l2 = 4 * q.numel() * 2 <= l2_bytes
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_l2 else None
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    h_start = time.perf_counter()
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(h_start, time.perf_counter())
    clocks.stop()
    barrier(world)
    st = fa.fa_get_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after timed region: {fa.fa_status_string(st)}")
    last = len(stages)
    ms_total = (sum(e[0].elapsed_time(e[last]) for e in evs) if flush is not None
                else t_start.elapsed_time(t_end))
    ms_total = max_over_ranks(ms_total, world)
    stage_ms = {s: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, s in enumerate(stages)}
    ms_step = ms_total / args.steps
    value = (f_fwd + f_bwd) * world / (ms_step * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers: pinned host inputs in, pinned
    # host outputs (O, LSE, dQ, dK, dV) out, copies overlapped with compute over head chunks
    e2e = None
    if not args.no_e2e:
        from exact_io_aware_fwd_gb300.pipeline import HostAttention, VarlenHostAttention

        hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
        if varlen:
            ha = VarlenHostAttention(extra, H, d, device=dev, Hkv=k.shape[1])
            h2d, d2h = ha.transfer_bytes()

            def e2e_step():
                ha.run(hq, hk, hv, hdo, causal=w.causal, scale=w.scale, out=hout,
                       deterministic=det, graph=True)
        else:
            ha = HostAttention(B, H, N, d, device=dev, Hkv=k.shape[1])
            h2d, d2h = ha.transfer_bytes(with_kv=kv is not None)

            def e2e_step():
                ha.run(hq, hk, hv, hdo, causal=w.causal, scale=w.scale, kv_lens=kv, out=hout,
                       deterministic=det, block_index=index, graph=True)
        hout = {"O": torch.empty(q.shape, dtype=torch.bfloat16).pin_memory(),
                "dQ": torch.empty(q.shape, dtype=torch.bfloat16).pin_memory(),
                "dK": torch.empty(k.shape, dtype=torch.bfloat16).pin_memory(),
                "dV": torch.empty(k.shape, dtype=torch.bfloat16).pin_memory(),
                "LSE": torch.empty(lse_shape, dtype=torch.float32).pin_memory()}

        for _ in range(2):
            e2e_step()
        link = host_link_gbs(hq, hout["O"], stream)
        barrier(world)
        torch.cuda.synchronize()
        # one event per replay boundary: the total and each replay's own duration
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        marks[0].record(stream)
        for i in range(args.steps):
            e2e_step()
            marks[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        per = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
        e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), world) / args.steps
        # what bounds a step: the device time of the same work, the copies at the measured link
        # rates (both directions at once), and the pipeline's fill and drain (the first chunk's
        # inputs and the last chunk's outputs, which nothing overlaps)
        n_ch = len(ha.plan)
        copies_ms = (h2d + d2h) / (link["both"] * 1e6)
        fill_drain_ms = (h2d / n_ch) / (link["h2d"] * 1e6) + (d2h / n_ch) / (link["d2h"] * 1e6)
        bound_ms = max(ms_step, copies_ms) + fill_drain_ms
        e2e = {"value": (f_fwd + f_bwd) * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "replay_ms": {"median": statistics.median(per), "min": min(per), "max": max(per)},
               "chunks": n_ch, "host_link_gbs": link,
               "bound_ms": {"device_step": ms_step, "copies_both_directions": copies_ms,
                            "fill_and_drain": fill_drain_ms, "bound": bound_ms},
               "median_over_device_step": statistics.median(per) / ms_step}
        assert fa.fa_get_error() == fa.FA_OK

    if rank != 0:
        return

    # ---- roofline of the dominant kernel (largest share of the step)
    peaks, src = load_peaks()
    bwd_stage = "bwd" if two_stage else "bwd_dkdv"
    dom = max(("fwd", bwd_stage), key=lambda s: stage_ms[s])
    dom_flops = f_fwd if dom == "fwd" else f_bwd
    achieved = dom_flops / (stage_ms[dom] * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    bwd_call = ("fa_bwd_varlen" if varlen else "fa_bwd_gqa" if gqa else
                "fa_bwd_block_sparse" if index is not None else "fa_bwd_deterministic")
    kernel_name = {"fwd": "fwd_kernel", "bwd_dkdv": "bwd_dkdv_kernel", "bwd": bwd_call}[dom]
    roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"bf16_tflops (burst) of {src}",
                "traffic": recorded_traffic(kernel_name, w.name)}

    cpu = None
    if not args.no_cpu_baseline:
        flops_s, dt, sample = time_oracle_once(w, q, k, v, do, extra, min_seconds=10.0)
        cpu = {"value": flops_s / dt / 1e12, "unit": "TFLOPS", "cores": cpu_cores(),
               "kind": "oracle", "sample": sample, "seconds": dt,
               "full_step_seconds_extrapolated": (f_fwd + f_bwd) / (flops_s / dt)}

    fwd_tf = f_fwd / (stage_ms["fwd"] * 1e-3) / 1e12
    bwd_ms = sum(stage_ms[s] for s in stages[1:])
    effective = None
    if w.kv_len_range is not None:  # the work the kernels do: only the visible (query, key) pairs
        e_fwd, e_bwd = w.flops_effective(kv)
        effective = {"note": "FLOPs of the visible (query, key) pairs, N * len_b per head",
                     "tflops": (e_fwd + e_bwd) * world / (ms_step * 1e-3) / 1e12,
                     "fwd_tflops": e_fwd / (stage_ms["fwd"] * 1e-3) / 1e12,
                     "bwd_tflops": e_bwd / (bwd_ms * 1e-3) / 1e12,
                     "fraction_of_nominal": (e_fwd + e_bwd) / (f_fwd + f_bwd)}
        effective["fwd_frac_of_peak"] = effective["fwd_tflops"] / peak
        effective["bwd_frac_of_peak"] = effective["bwd_tflops"] / peak
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, extra, args, world),
        "l2": ("flushed: 256 MB written between steps, outside the per-step events summed"
               if in_l2 else "inputs larger than L2 (no flush)"),
        "fwd_tflops": fwd_tf, "fwd_frac_of_peak": fwd_tf / peak,
        "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
        "bwd_frac_of_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / peak,
        "stage_ms": stage_ms,
        "effective": effective,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.ingest_ncu:
        ingest_ncu(args.ingest_ncu, args.workload, args.ncu_command)
        return
    w = BY_NAME[args.workload]
    if args.heads is not None:
        from dataclasses import replace

        w = replace(w, H=args.heads, name=f"{w.name}[H={args.heads}]")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
