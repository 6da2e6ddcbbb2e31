"""Build libemufp8.so (the GEMM library) and libemupeaks.so (the instruction-rate
microbenchmark bench.py divides by) in-tree with nvcc for sm_103a (GB300).

    python -m bit_exact_fp8_gb300.build [--force]

One translation unit per library, one -gencode, no cmake; the two compile in
parallel, and each is rebuilt only when one of its sources or headers is newer.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libemufp8.so")
PEAKS_LIB = os.path.join(PKG, "libemupeaks.so")
SOURCES = [os.path.join(CSRC, "emu_api.cu")]
PEAKS_SOURCES = [os.path.join(CSRC, "emu_peaks.cu")]
PEAKS_DEPS = PEAKS_SOURCES + [os.path.join(INCLUDE, "emu_peaks.h")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] \
    + [os.path.join(INCLUDE, "emu_fp8.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libemufp8")


def _up_to_date(lib: str, deps) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in deps)


def up_to_date() -> bool:
    return _up_to_date(LIB, DEPS) and _up_to_date(PEAKS_LIB, PEAKS_DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile whichever of the two libraries is stale; returns the GEMM library's path."""
    jobs = []
    for lib, srcs, deps in ((LIB, SOURCES, DEPS), (PEAKS_LIB, PEAKS_SOURCES, PEAKS_DEPS)):
        if force or not _up_to_date(lib, deps):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc_path()] + NVCC_FLAGS + srcs + ["-o", tmp]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            jobs.append((lib, tmp, subprocess.Popen(cmd)))
    failed = [lib for lib, _, proc in jobs if proc.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, f"nvcc ({', '.join(failed)})")
    for lib, tmp, _ in jobs:
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
