"""Builds libfa_sm103.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units are compiled in parallel into ``<repo>/_build`` and linked into
``exact_io_aware_fwd_gb300/libfa_sm103.so``.  A rebuild happens only when a source or header is
newer than the library (or when ``force=True``).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libfa_sm103.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_dq.cu", "fa_block_sparse.cu", "fa_noalloc.cu"]
HEADERS = [os.path.join(CSRC, "sm103.cuh"), os.path.join(CSRC, "fa_internal.h"),
           os.path.join(ROOT, "include", "fa.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          defines: dict | None = None, out_path: str | None = None) -> str:
    """Compile and link the library; returns its path.

    ``defines`` (name -> value) are passed as -D flags (the kernels' tuning parameters) and
    ``out_path`` places the library elsewhere than the package directory.
    """
    nvcc = _nvcc()
    lib_path = out_path or LIB_PATH
    tag = "" if not defines else "_" + "_".join(f"{k}{v}" for k, v in sorted(defines.items()))
    build_dir = os.path.join(BUILD_DIR, tag.strip("_") or "default")
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(lib_path, srcs + HEADERS + [__file__]):
        return lib_path
    objs = [os.path.join(build_dir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    extra += [f"-D{k}={v}" for k, v in (defines or {}).items()]

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    for cmd, r in results:
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("linking libfa_sm103.so failed")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
