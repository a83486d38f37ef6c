"""Build libssmscan.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "ssmscan.cu")
HDR = os.path.join(ROOT, "include", "ssmscan.h")
LIB = os.path.join(PKG, "libssmscan.so")
PEAKS_SRC = os.path.join(PKG, "csrc", "pipe_peaks.cu")
PEAKS_HDR = os.path.join(ROOT, "include", "pipe_peaks.h")
PEAKS_LIB = os.path.join(PKG, "libpipepeaks.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"),
    "-Xptxas", "-warn-spills",
]


def _compile(src, hdr, lib, force, verbose, extra):
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr), os.path.getmtime(__file__))
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    cmd = [NVCC, *FLAGS, *extra, src, "-o", lib]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    return lib


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile libssmscan.so (and the pipe-peak microbenchmark library used by
    the benchmark) if missing or older than their sources."""
    _compile(PEAKS_SRC, PEAKS_HDR, PEAKS_LIB, force, verbose, ())
    return _compile(SRC, HDR, LIB, force, verbose, extra)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
