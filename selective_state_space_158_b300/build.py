"""Builds libsscan.so (and the rate-probe library libsscan_peaks.so) in-tree with nvcc for
sm_103a (B300)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libsscan.so")
# Issue-rate microbenchmarks (the compute rooflines' denominators); not part of the scan library.
PEAKS_LIB = os.path.join(PKG, "libsscan_peaks.so")
PEAKS_SOURCES = ["sscan_peaks.cu"]
SOURCES = ["sscan_api.cu", "sscan_kernels.cu", "sscan_noalloc.cu", "sscan_conv.cu",
           "sscan_bwd.cu"]
HEADERS = ["sscan_device.cuh", "sscan_internal.h"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-Xptxas", "-warn-spills",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str, sources) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in list(sources) + HEADERS]
    deps += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(lib: str, sources, verbose: bool, extra_flags) -> None:
    tmp = lib + ".tmp"
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"),
           "-o", tmp, *[os.path.join(CSRC, f) for f in sources]]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile the library (and the rate probes) if any source is newer; returns the .so path."""
    if force or _stale(LIB, SOURCES):
        _compile(LIB, SOURCES, verbose, extra_flags)
    if force or _stale(PEAKS_LIB, PEAKS_SOURCES):
        _compile(PEAKS_LIB, PEAKS_SOURCES, verbose, extra_flags)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
