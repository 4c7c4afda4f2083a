"""Build libnvfp4.so in-tree with nvcc for sm_103a (B300).

Usage: python -m nvfp4_precision_02_b300.build [--force] [--verbose]
The CUDA runtime is linked statically, so loading the library needs only the
NVIDIA driver (and nothing at all on a machine without a GPU, where every
entry point returns NVFP4_ERR_DEVICE after argument validation).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC_DIR = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libnvfp4.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _sources():
    out = []
    for d in (SRC_DIR, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                out.append(os.path.join(d, f))
    return out


def nvcc_command(out: str = LIB, verbose: bool = False):
    cmd = ["nvcc", *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
           "-cudart", "static", "-I", INCLUDE, "-o", out, os.path.join(SRC_DIR, "nvfp4.cu"), "-ldl", "-lpthread",
           "-lrt"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    stale = (not os.path.exists(LIB)) or any(os.path.getmtime(s) > os.path.getmtime(LIB) for s in _sources())
    if force or stale:
        tmp = LIB + ".tmp"
        subprocess.check_call(nvcc_command(tmp, verbose))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB)
