"""bench.py's multi-process path on the CPU: two gloo ranks launched by torchrun run the
reference (oracle) arm; rank 0 alone prints one JSON line and every rank exits 0."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_two_ranks_gloo():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29533", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "smoke-1x1x128x64"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["full_step_seconds_extrapolated"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["n_gpus"] == 2 and d["config"]["parallelism"] == "replicas x2"
    # the same config object as the CUDA arm's line for these arguments (both arms build it with
    # bench.workload_config); how the arm treats L2 is a key of its own, outside config
    import argparse
    import importlib.util

    from exact_io_aware_fwd_gb300.workloads import BY_NAME, workload_inputs

    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    w = BY_NAME["smoke-1x1x128x64"]
    extra = workload_inputs(w)[4]
    assert d["config"] == bench.workload_config(w, extra, argparse.Namespace(bwd="atomic"), 2)
    assert "l2" not in d["config"] and d["l2"]


def test_max_over_ranks_gloo(tmp_path):
    """The timing reduction used by bench.py: the max of the ranks' times."""
    script = tmp_path / "ranks.py"
    script.write_text(
        "import sys, torch.distributed as dist\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "dist.init_process_group('gloo')\n"
        "r = dist.get_rank()\n"
        "m = bench.max_over_ranks(1.0 + r, 2)\n"
        "assert m == 2.0, m\n"
        "bench.barrier(2)\n"
        "dist.destroy_process_group()\n")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29534", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]


def test_cpu_baseline_sample_for_every_workload_kind():
    """bench.py's oracle sample works for dense, key-padded, block-sparse, GQA and packed
    variable-length workloads (small copies of each kind)."""
    import dataclasses
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from exact_io_aware_fwd_gb300.workloads import BY_NAME, workload_inputs

    small = {"long-causal-1x32x16384x128": dict(H=1, N=300),
             "ragged-8x12x2000x128": dict(B=2, H=1, N=300, kv_len_range=(100, 300)),
             "butterfly-1x32x16384x128": dict(H=1, N=300),
             "gqa-1x32kv8x16384x128": dict(H=4, Hkv=2, N=300),
             "varlen-16x16x512-4096x128": dict(B=3, H=2, N=300, seqlen_range=(50, 300))}
    for name, kw in small.items():
        w = dataclasses.replace(BY_NAME[name], **kw)
        q, k, v, do, extra = workload_inputs(w)
        flops, dt, sample = bench.time_oracle_once(w, q, k, v, do, extra)
        assert flops > 0 and dt > 0 and sample, name
