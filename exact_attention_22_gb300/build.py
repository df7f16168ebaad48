"""Build the sm_103a CUDA library in-tree: exact_attention_22_gb300/libfa.so.

Three translation units (the forward pass, the backward pass and the
host-buffer entry point), compiled in parallel with nvcc directly (no cmake, no torch extension machinery) and
linked into one shared library.  One -gencode; nvcc cross-compiles, so this
works without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SRCS = [os.path.join(CSRC, "fa_fwd.cu"), os.path.join(CSRC, "fa_bwd.cu"), os.path.join(CSRC, "fa_host_io.cu")]
DEPS = SRCS + [os.path.join(CSRC, "sm103_ptx.cuh"), os.path.join(CSRC, "fa_host.cuh"),
               os.path.join(ROOT, "include", "fa.h")]
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
    tag = "%d" % os.getpid()
    objs = [os.path.join(CSRC, os.path.basename(s)[:-3] + "." + tag + ".o") for s in SRCS]
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-I" + os.path.join(ROOT, "include"), "-Xcompiler", "-fPIC"]
    if verbose:
        flags.append("-Xptxas=-v")
    procs = [subprocess.Popen([nvcc()] + flags + ["-c", "-o", o, s]) for s, o in zip(SRCS, objs)]
    rcs = [pr.wait() for pr in procs]
    try:
        for s, rc in zip(SRCS, rcs):
            if rc != 0:
                raise subprocess.CalledProcessError(rc, "nvcc -c " + s)
        tmp = LIB + ".tmp" + tag
        subprocess.check_call([nvcc(), ARCH, "-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
