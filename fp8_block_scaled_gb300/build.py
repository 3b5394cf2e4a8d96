"""Build step of the CUDA library: nvcc for sm_103a, in-tree.

Produces ``fp8_block_scaled_gb300/_build/libfp8bs.so`` from the sources in
``csrc/`` with ``-gencode arch=compute_103a,code=sm_103a``.  The CUDA runtime
is linked statically; the driver API (tensor-map encoding) is reached through
the runtime's driver entry-point query, so no libcuda link is needed.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libfp8bs.so")
SOURCES = ["fp8bs_api.cu"]
HEADERS = ["ptx.cuh", "grouped_gemm.cuh", "grouped_gemm_pair.cuh", "grouped_gemm_promote.cuh"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _inputs():
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "fp8bs.h"))
    paths.append(os.path.abspath(__file__))
    return paths


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if missing or older than any of its sources."""
    if not force and not is_stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-I", INCLUDE, "-I", CSRC, "-o", tmp]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
