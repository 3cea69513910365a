"""The L2 fp32-reduction throughput microbenchmark (tests/csrc/l2_reduction_rate.cu) builds, runs
without a CUDA error, and reports a plausible GPU-wide rate for both forms (more than 1 TB/s)."""

import os
import re
import subprocess

import pytest

from exact_io_aware_fwd_gb300 import build_lib

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_l2_reduction_rate(tmp_path):
    exe = tmp_path / "l2_reduction_rate"
    subprocess.run([build_lib._nvcc(), *build_lib.ARCH, "-O3", "-std=c++17", "-I", build_lib.CSRC,
                    os.path.join(HERE, "csrc", "l2_reduction_rate.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout
    rates = [float(m) for m in re.findall(r": ([0-9.]+) GB/s", out)]
    assert len(rates) == 6, out
    assert all(r > 1000.0 for r in rates), out
