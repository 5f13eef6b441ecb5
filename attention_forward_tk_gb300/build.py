"""Compile the CUDA library in-tree: ``_build/libtk_attn.so`` for sm_103a.

Two translation units (host launcher + kernels; the host-buffer pipeline),
one ``-gencode``; no cmake.
The same command works on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
CSRC = os.path.join(_HERE, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libtk_attn.so")
SOURCES = [os.path.join(CSRC, "tk_attn.cu"), os.path.join(CSRC, "tk_attn_host.cpp")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
    os.path.join(INCLUDE, "tk_attn.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
    "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build libtk_attn.so if it is missing or older than its sources."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in DEPS if os.path.exists(p))
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = f"{LIB}.tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building libtk_attn.so")
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
