"""Build the sm_103a CUDA library in-tree: exact_attention_22_gb300/libfa.so.

One translation unit, one -gencode, compiled with nvcc directly (no cmake, no
torch extension machinery).  nvcc cross-compiles, so this works without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "fa_fwd.cu")
DEPS = [SRC, os.path.join(PKG, "csrc", "sm103_ptx.cuh"), os.path.join(ROOT, "include", "fa.h")]
LIB = os.path.join(PKG, "libfa.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def build(force: bool = False, verbose: bool = False) -> str:
    stale = not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(p) for p in DEPS)
    if not (force or stale):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-I" + os.path.join(ROOT, "include"),
           "-shared", "-Xcompiler", "-fPIC", "-o", tmp, SRC]
    if verbose:
        cmd.insert(2, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
