"""The boundary is usable from plain C: a C99 program compiled with gcc -pedantic against
include/fa.h alone links libfa_sm103.so and gets the documented answers from the calls that
need no GPU."""

import os
import shutil
import subprocess

import pytest

import exact_io_aware_fwd_gb300 as fa
from exact_io_aware_fwd_gb300.build_lib import LIB_PATH

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c99_client_links_and_runs(tmp_path):
    fa.build()
    exe = tmp_path / "client"
    libdir = os.path.dirname(LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "csrc", "c_abi_client.c"), "-o", str(exe),
                    "-L", libdir, "-l:" + os.path.basename(LIB_PATH), "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                         timeout=60).stdout.splitlines()
    got = dict(line.split(" ", 1) for line in out)
    assert got["status_string"] == "device pipeline wait timed out"
    assert int(got["workspace"]) == 128 * 64 * 4 + 2 * 512 + 256  # + one 16-byte tile record
    assert int(got["unsupported"]) == fa.FA_ERR_UNSUPPORTED
    assert int(got["invalid"]) == fa.FA_ERR_INVALID_ARG
