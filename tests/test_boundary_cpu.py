"""The C ABI without a GPU: the library builds and loads, exports what
include/fa.h declares, and rejects bad arguments before touching CUDA."""
import math
import os
import re
import shutil
import subprocess

import pytest

import exact_attention_22_gb300 as fa
from exact_attention_22_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def _declared():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fa_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert {"fa_fwd", "fa_get_device_status", "fa_status_string"} <= declared
    out = subprocess.check_output(["nm", "-D", "--defined-only", fa.library_path()], text=True)
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    assert declared <= exported, declared - exported


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# Fake but 16-byte-aligned, non-overlapping "device" addresses: every call
# below must fail validation before any CUDA call is made.
GOOD = dict(q=1 << 20, k=2 << 20, v=3 << 20, o=4 << 20, lse=5 << 20, B=1, H=2, N=256, D=64,
            scale=0.125, causal=0, dtype=0, stream=0)


def _call(**kw):
    a = dict(GOOD, **kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["scale"],
                     a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(D=32), 2), (dict(D=256), 2),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1),
    (dict(causal=2), 1), (dict(dtype=2), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=math.inf), 1), (dict(scale=math.nan), 1),
    (dict(q=0), 3), (dict(o=0), 3), (dict(lse=0), 3), (dict(k=(2 << 20) + 8), 3), (dict(v=(3 << 20) + 2), 3),
    (dict(o=(1 << 20) + 4096), 1),           # output overlaps q
    (dict(lse=(4 << 20) + 64), 1),           # lse overlaps o
    (dict(B=1 << 16, H=1 << 16), 1),         # B*H does not fit the grid
])
def test_argument_errors(lib, kw, status):
    assert _call(**kw) == status


def test_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.attention(x, x, x)


def test_splitkv_workspace_size(lib):
    assert fa.fa_splitkv_workspace_bytes(2, 3, 100, 128, 5) == 5 * 2 * 3 * 100 * (4 * 128 + 16)
    for bad in ((0, 1, 1, 64, 1), (1, 1, 1, 96, 1), (1, 1, 1, 64, 0), (1, 1, 1, 64, 65)):
        assert fa.fa_splitkv_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("splits,ws,ws_bytes,status", [
    (0, 6 << 20, 1 << 20, 1), (65, 6 << 20, 1 << 20, 1),
    (4, 6 << 20, 16, 1),                     # too small
    (4, 0, 1 << 20, 3), (4, (6 << 20) + 4, 1 << 20, 3),
    (4, (4 << 20) - 1024, 1 << 20, 1),       # overlaps o
])
def test_splitkv_argument_errors_without_gpu(lib, splits, ws, ws_bytes, status):
    a = GOOD
    assert fa.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["scale"],
                             a["causal"], a["dtype"], splits, ws, ws_bytes, 0) == status


@pytest.mark.parametrize("kw,splits,status", [
    (dict(), 0, 1), (dict(), 65, 1),
    (dict(D=96), 4, 2), (dict(B=0), 4, 1), (dict(N=0), 4, 1), (dict(causal=2), 4, 1), (dict(dtype=2), 4, 1),
    (dict(scale=0.0), 4, 1), (dict(scale=math.nan), 4, 1),
    (dict(q=0), 4, 3), (dict(v=(3 << 20) + 2), 4, 3), (dict(lse=(5 << 20) + 4), 4, 3),
    (dict(o=(1 << 20) + 4096), 4, 1),        # output overlaps q
])
def test_noalloc_argument_errors_without_gpu(lib, kw, splits, status):
    """Every argument is checked before the scratch buffer's address is looked
    up (without a GPU any CUDA call would give FA_ERR_CUDA instead)."""
    a = dict(GOOD, **kw)
    assert fa.fa_fwd_splitkv_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                                     a["scale"], a["causal"], a["dtype"], splits, 0) == status


def test_fault_selftests_check_arguments_without_gpu(lib):
    a = GOOD
    assert fa.fa_selftest_fwd_fault(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                                    a["scale"], a["causal"], a["dtype"], -1, 0) == 1
    assert fa.fa_selftest_fwd_fault(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], 96,
                                    a["scale"], a["causal"], a["dtype"], 3, 0) == 2
    ptr = [(i + 1) << 20 for i in range(10)]
    assert fa.fa_selftest_bwd_fault(*ptr[:9], 1, 2, 256, 64, 0.125, 0, 0, ptr[9], 1 << 20, -1, 0) == 1
    assert fa.fa_selftest_bwd_fault(*ptr[:9], 1, 2, 256, 96, 0.125, 0, 0, ptr[9], 1 << 20, 2, 0) == 2


@pytest.mark.parametrize("H,H_kv,status", [(6, 4, 1), (6, 0, 1), (6, -2, 1), (4, 8, 1)])
def test_gqa_head_count_errors(lib, H, H_kv, status):
    a = GOOD
    assert fa.fa_fwd_gqa(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, H, H_kv, 256, 64, 0.125, 0, 0, 0) == status


def test_bwd_workspace_size(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    assert fa.fa_bwd_workspace_bytes(2, 3, 100, 128) == r256(600 * 128 * 4) + r256(600 * 4)
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 64) == 256 + 256
    for bad in ((0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 96)):
        assert fa.fa_bwd_workspace_bytes(*bad) == 0


# Fake aligned addresses 1 MiB apart (each tensor of B1 H2 N256 D64 is 64 KiB).
BWD = dict(q=1 << 20, k=2 << 20, v=3 << 20, o=4 << 20, dout=5 << 20, lse=6 << 20, dq=7 << 20, dk=8 << 20,
           dv=9 << 20, ws=10 << 20, ws_bytes=1 << 20, B=1, H=2, N=256, D=64, scale=0.125, causal=1, dtype=0)


def _bwd(**kw):
    a = dict(BWD, **kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"], a["H"],
                     a["N"], a["D"], a["scale"], a["causal"], a["dtype"], a["ws"], a["ws_bytes"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(D=256), 2),
    (dict(B=0), 1), (dict(N=-3), 1), (dict(causal=2), 1), (dict(dtype=5), 1),
    (dict(scale=0.0), 1), (dict(scale=math.nan), 1),
    (dict(dq=0), 3), (dict(lse=0), 3), (dict(ws=0), 3), (dict(dout=(5 << 20) + 8), 3), (dict(ws=(10 << 20) + 4), 3),
    (dict(ws_bytes=1024), 1),                  # workspace too small
    (dict(dq=(1 << 20) + 1024), 1),            # dq overlaps q
    (dict(dk=(9 << 20) - 4096), 1),            # dk overlaps dv
    (dict(ws=(6 << 20) - 256), 1),             # workspace overlaps lse
    (dict(dv=(4 << 20) + 16), 1),              # dv overlaps o
])
def test_bwd_argument_errors_without_gpu(lib, kw, status):
    assert _bwd(**kw) == status


def test_bwd_binding_rejects_bad_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError):
        fa.attention_backward(x, x, x, x, lse, x)


FP8 = dict(q=1 << 20, k=2 << 20, vt=3 << 20, qs=4 << 20, ks=5 << 20, vs=6 << 20, o=7 << 20, lse=8 << 20,
           B=1, H=2, N=256, D=128, scale=0.09, causal=1)


def _fp8(**kw):
    a = dict(FP8, **kw)
    return fa.fa_fwd_fp8(a["q"], a["k"], a["vt"], a["qs"], a["ks"], a["vs"], a["o"], a["lse"], a["B"], a["H"],
                         a["N"], a["D"], a["scale"], a["causal"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), 2), (dict(D=96), 2),
    (dict(N=100), 1), (dict(N=0), 1), (dict(B=0), 1), (dict(causal=3), 1), (dict(scale=-1.0), 1),
    (dict(q=0), 3), (dict(vs=0), 3), (dict(ks=(5 << 20) + 4), 3), (dict(lse=(8 << 20) + 8), 3),
    (dict(o=(1 << 20) + 4096), 1),            # o overlaps q
    (dict(lse=(7 << 20) + 1024), 1),          # lse overlaps o
    (dict(o=(4 << 20) - 64 * 1024), 1),       # o overlaps the Q scales
])
def test_fp8_argument_errors_without_gpu(lib, kw, status):
    assert _fp8(**kw) == status


def test_host_workspace_size(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    t = 2 * 3 * 100 * 128 * 2
    assert fa.fa_fwd_host_workspace_bytes(2, 3, 100, 128) == 4 * r256(t) + r256(2 * 3 * 100 * 4)
    for bad in ((0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 96)):
        assert fa.fa_fwd_host_workspace_bytes(*bad) == 0


HOST = dict(q=1 << 20, k=2 << 20, v=3 << 20, o=4 << 20, lse=5 << 20, ws=6 << 20, ws_bytes=1 << 20,
            B=1, H=2, N=256, D=64, scale=0.125, causal=1, dtype=0)


def _host(**kw):
    a = dict(HOST, **kw)
    return fa.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["scale"],
                          a["causal"], a["dtype"], a["ws"], a["ws_bytes"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(B=0), 1), (dict(causal=2), 1), (dict(dtype=3), 1), (dict(scale=math.inf), 1),
    (dict(q=0), 3), (dict(lse=(5 << 20) + 4), 3), (dict(ws=(6 << 20) + 16), 3),   # workspace needs 256 bytes
    (dict(ws_bytes=4096), 1),
    (dict(o=(1 << 20) + 1024), 1),            # o overlaps q
    (dict(), 1),                              # fake addresses are not page-locked host memory
])
def test_host_argument_errors_without_gpu(lib, kw, status):
    assert _host(**kw) == status


def test_host_binding_rejects_device_or_pageable_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float16)   # pageable
    with pytest.raises(ValueError):
        fa.attention_host(x, x, x)


def test_bwd_host_workspace_size(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    t = 2 * 3 * 100 * 64 * 2
    # one chunk here (small problem): fa_bwd's workspace for all 6 planes
    assert fa.fa_bwd_host_workspace_bytes(2, 3, 100, 64) == 8 * r256(t) + r256(600 * 4) + \
        fa.fa_bwd_workspace_bytes(1, 6, 100, 64)
    for bad in ((0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 96)):
        assert fa.fa_bwd_host_workspace_bytes(*bad) == 0


BWDH = dict(q=1 << 20, k=2 << 20, v=3 << 20, o=4 << 20, dout=5 << 20, lse=6 << 20, dq=7 << 20, dk=8 << 20,
            dv=9 << 20, ws=10 << 20, ws_bytes=4 << 20, B=1, H=2, N=256, D=64, scale=0.125, causal=1, dtype=0)


def _bwd_host(**kw):
    a = dict(BWDH, **kw)
    return fa.fa_bwd_host(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                          a["H"], a["N"], a["D"], a["scale"], a["causal"], a["dtype"], a["ws"], a["ws_bytes"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(N=0), 1), (dict(causal=2), 1), (dict(scale=0.0), 1),
    (dict(dq=0), 3), (dict(ws=(10 << 20) + 16), 3), (dict(ws_bytes=1024), 1),
    (dict(dq=(1 << 20) + 1024), 1),           # dq overlaps q
    (dict(dk=(9 << 20) - 4096), 1),           # dk overlaps dv
    (dict(), 1),                              # fake addresses are not page-locked host memory
])
def test_bwd_host_argument_errors_without_gpu(lib, kw, status):
    assert _bwd_host(**kw) == status


@pytest.mark.parametrize("args", [(0, 32, 8, 1, 4096, 128, 1), (1, 32, 6, 1, 4096, 128, 1), (1, 32, 8, 1, 4096, 96, 1),
                                  (1, 32, 8, 8, 4, 128, 1), (1, 32, 8, 1, 4096, 128, 2)])
def test_kv_splits_hint_rejects_invalid_sizes(lib, args):
    assert fa.fa_fwd_kv_splits_hint(*args) == -1


def test_fp8_host_workspace_size_and_errors(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    e = 2 * 3 * 256 * 128
    sc = 2 * 3 * 2 * 4
    assert fa.fa_fwd_fp8_host_workspace_bytes(2, 3, 256, 128) == 3 * r256(e) + 3 * r256(sc) + r256(2 * e) + \
        r256(2 * 3 * 256 * 4)
    for bad in ((0, 1, 16, 128), (1, 1, 100, 128), (1, 1, 256, 64)):
        assert fa.fa_fwd_fp8_host_workspace_bytes(*bad) == 0
    a = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 6 << 20, 7 << 20, 8 << 20]
    call = lambda N=256, D=128, ws=10 << 20, wsb=64 << 20: fa.fa_fwd_fp8_host(*a, 1, 2, N, D, 0.09, 1, ws, wsb, 0)
    assert call(D=64) == 2
    assert call(N=100) == 1
    assert call(ws=(10 << 20) + 16) == 3
    assert call(wsb=1024) == 1
    assert call() == 1          # fake addresses are not page-locked host memory


@pytest.mark.parametrize("H,H_kv,status", [(6, 4, 1), (6, 0, 1), (4, 8, 1)])
def test_bwd_gqa_head_count_errors(lib, H, H_kv, status):
    a = dict(BWD)
    assert fa.fa_bwd_gqa(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], 1, H, H_kv,
                         256, 64, 0.125, 1, 0, a["ws"], a["ws_bytes"], 0) == status


C_PROGRAM = r"""
#include <stdio.h>
#include "fa.h"

int main(void) {
    size_t ws = fa_splitkv_workspace_bytes(1, 2, 256, 64, 4);
    size_t bw = fa_bwd_workspace_bytes(1, 2, 256, 64);
    int st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 0, 2, 256, 64, 0.125f, 0, FA_FP16, (cudaStream_t)0);
    int st2 = fa_fwd((void*)16, (void*)32, (void*)48, (void*)64, (float*)80, 1, 2, 256, 96, 0.125f, 0, FA_FP16,
                     (cudaStream_t)0);
    printf("%zu %zu %d %d %s\n", ws, bw, st, st2, fa_status_string(st));
    return 0;
}
"""


def test_header_is_plain_c(lib, tmp_path):
    """include/fa.h compiles as C99 with warnings as errors, and a C program
    linked against the library gets the sizes and argument errors the binding
    sees (both returned before anything reaches CUDA)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "prog.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "prog"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    libpath = fa.library_path()
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                    cuda_inc, str(src), libpath, "-Wl,-rpath," + os.path.dirname(libpath), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == fa.fa_splitkv_workspace_bytes(1, 2, 256, 64, 4)
    assert int(out[1]) == fa.fa_bwd_workspace_bytes(1, 2, 256, 64)
    assert int(out[2]) == 1 and out[4] == "FA_ERR_INVALID_ARG"   # B = 0
    assert int(out[3]) == 2                                     # D = 96: unsupported


def test_wrapper_output_checks():
    """The wrappers' checks of caller-provided outputs and workspaces (the C ABI
    sees only pointers): exact shape and dtype, contiguous, right device or
    page-locked memory; a workspace must be device memory."""
    import torch
    from exact_attention_22_gb300 import binding as b

    cpu = torch.device("cpu")
    t = torch.empty(2, 3, 4)
    b._check_given(None, (9,), torch.float16, "out", cpu)
    b._check_given(t, (2, 3, 4), torch.float32, "out", cpu)
    for bad, shape, dtype in ((t, (2, 3, 5), torch.float32), (t, (2, 3, 4), torch.float16),
                              (t.transpose(0, 1), (3, 2, 4), torch.float32)):
        with pytest.raises(ValueError, match="out"):
            b._check_given(bad, shape, dtype, "out", cpu)
    with pytest.raises(ValueError, match="lse"):
        b._check_given(t, (2, 3, 4), torch.float32, "lse", pinned=True)   # pageable host memory
    with pytest.raises(ValueError, match="workspace"):
        b._check_workspace(torch.empty(16, dtype=torch.uint8), cpu)
    b._same_device((t, t))
