"""Builds libnvfp4.so (the C-ABI library, sm_103a) in-tree with nvcc.

Usage: python -m nvfp4_gemm_act_b300.build [--verbose]
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libnvfp4.so")
# the same sources with the index checks of the kernels compiled in (-DNVFP4_DEBUG)
DEBUG_LIB = os.path.join(HERE, "libnvfp4_debug.so")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "attention.cu", "noalloc.cu", "mma_probe.cu"]
HEADERS = ["nvfp4_device.cuh", "nvfp4_internal.h", "pointer_check.h"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-Xptxas", "-v",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "nvfp4.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (``debug``: the index-checking build) if a source is newer than it.
    Returns the .so path."""
    lib = DEBUG_LIB if debug else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + ".tmp"
    flags = NVCC_FLAGS + (["-DNVFP4_DEBUG"] if debug else [])
    cmd = [_nvcc(), *flags, "-o", tmp, *[os.path.join(CSRC, f) for f in SOURCES]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
    print(build(force=True, verbose="--verbose" in sys.argv, debug=True))
