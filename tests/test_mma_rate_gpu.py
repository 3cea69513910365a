"""The tcgen05.mma issue-rate microbenchmark (tests/csrc/mma_issue_rate.cu) builds, runs without a
CUDA error or pipeline timeout, and sees the tensor core's rate: at N >= 128 one M = 128, K = 16
MMA per 64 cycles on an otherwise idle sub-partition (8,192 FLOP/clk/SM), allowing 25% slack."""

import os
import re
import subprocess

import pytest

from exact_io_aware_fwd_gb300 import build_lib

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_mma_issue_rate(tmp_path):
    exe = tmp_path / "mma_issue_rate"
    subprocess.run([build_lib._nvcc(), *build_lib.ARCH, "-O3", "-std=c++17", "-I", build_lib.CSRC,
                    os.path.join(HERE, "csrc", "mma_issue_rate.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout
    lines = out.strip().splitlines()
    assert len(lines) == 20, out
    for line in lines:
        assert "no error st=0" in line, line
    idle_128 = [ln for ln in lines if "N=128" in ln and "busy" not in ln]
    for ln in idle_128:
        cyc = float(re.search(r"complete ([0-9.]+) cyc/mma", ln).group(1))
        assert 60.0 <= cyc <= 80.0, ln
