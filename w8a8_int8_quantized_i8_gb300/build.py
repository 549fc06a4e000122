"""Builds libi8.so (the CUDA library behind include/i8.h) in-tree with nvcc,
and beside it libi8probe.so, a measurement helper for the benchmark (the
legacy warp MMA's int8 and fp16 rates; not part of the W8A8 path).

One translation unit each, one ``-gencode`` target (sm_103a), no cmake; the
two compile in parallel.  The outputs are git-ignored and rebuilt whenever a
source is newer than them.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libi8.so")
MAIN = os.path.join(CSRC, "i8_api.cu")
PROBE_LIB = os.path.join(PKG, "libi8probe.so")
PROBE_SRC = os.path.join(CSRC, "engine_probe.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    # IEEE fp32 behaviour (nvcc's defaults, stated so no flag set can drop
    # them): no flush to zero, correctly rounded division and square root
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-shared",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libi8")


def _sources():
    return ([s for s in glob.glob(os.path.join(CSRC, "*.cu")) if s != PROBE_SRC]
            + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "i8.h")])


def _stale(lib, sources) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources)


def stale() -> bool:
    return _stale(LIB, _sources()) or _stale(PROBE_LIB, [PROBE_SRC])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libi8.so and libi8probe.so if missing or older than their sources."""
    jobs = []
    for lib, src, sources in ((LIB, MAIN, _sources()), (PROBE_LIB, PROBE_SRC, [PROBE_SRC])):
        if force or _stale(lib, sources):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc(), *NVCC_FLAGS, "-o", tmp, src]
            if verbose:
                print(" ".join(cmd))
            jobs.append((subprocess.Popen(cmd), tmp, lib))
    failed = [lib for proc, _, lib in jobs if proc.wait() != 0]
    if failed:
        raise RuntimeError(f"nvcc failed building {', '.join(os.path.basename(f) for f in failed)}")
    for _, tmp, lib in jobs:
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
