"""The MUFU exponential throughput microbenchmark (tests/csrc/mufu_ex2_rate.cu) builds, runs
without a CUDA error, and reports a plausible rate for both forms (at least 4 exponentials per
cycle per SM)."""

import os
import re
import subprocess

import pytest

from exact_io_aware_fwd_gb300 import build_lib

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_mufu_ex2_rate(tmp_path):
    exe = tmp_path / "mufu_ex2_rate"
    subprocess.run([build_lib._nvcc(), *build_lib.ARCH, "-O3", "-std=c++17",
                    os.path.join(HERE, "csrc", "mufu_ex2_rate.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout
    rates = [float(m) for m in re.findall(r": ([0-9.]+) exponentials per cycle per SM", out)]
    assert len(rates) == 6, out
    assert all(r >= 4.0 for r in rates), out
