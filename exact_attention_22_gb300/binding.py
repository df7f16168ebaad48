"""ctypes binding of libfa.so: the same entry points as include/fa.h.

``fa_fwd`` / ``fa_get_device_status`` / ``fa_status_string`` take plain
integers (device pointers, sizes, a stream handle) exactly like the C ABI.
``attention`` is a convenience wrapper for torch CUDA tensors: it only checks
shapes, allocates the outputs with torch and passes pointers through.  Every
step of the computation runs in the CUDA library.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_FP16, FA_BF16 = 0, 1
FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
                4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_TOO_LARGE"}

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s returned %s" % (where, STATUS_NAMES.get(status, status)))
        self.status = status


def _check_given(t, shape, dtype, name, device=None, pinned=False):
    """A caller-provided output must be exactly what the kernel writes: its
    shape and dtype, contiguous, and on the inputs' device (or page-locked host
    memory for the host entry points).  The C ABI sees only a pointer."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError("%s must be %s %s" % (name, dtype, list(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if pinned:
        if t.is_cuda or not t.is_pinned():
            raise ValueError("%s must be a page-locked host tensor" % name)
    elif t.device != device:
        raise ValueError("%s must be on %s" % (name, device))


def _check_workspace(ws, device):
    """A caller-provided workspace: contiguous bytes on the given CUDA device
    (its size is checked by the library)."""
    if ws is None:
        return
    if not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on %s" % device)


def _same_device(ts):
    """Every tensor of a device call on one GPU: a pointer from another device
    would reach the kernel."""
    dev = ts[0].device
    if any(t.device != dev for t in ts[1:]):
        raise ValueError("all tensors must be on one device (%s)" % dev)


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libfa.so is not built (run exact_attention_22_gb300.build.build() or "
                               "__graft_entry__.build()); there is no fallback path")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, I, vp]
        lib.fa_fwd.restype = I
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = I
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, F, I, I, vp]
        lib.fa_fwd_gqa.restype = I
        lib.fa_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = I
        lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, I, I, vp]
        lib.fa_fwd_splitkv_noalloc.restype = I
        lib.fa_noalloc_scratch_bytes.argtypes = []
        lib.fa_noalloc_scratch_bytes.restype = ctypes.c_size_t
        lib.fa_selftest_wait_timeout.argtypes = [vp]
        lib.fa_selftest_wait_timeout.restype = I
        lib.fa_selftest_fwd_fault.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, I, I, vp]
        lib.fa_selftest_fwd_fault.restype = I
        lib.fa_selftest_bwd_fault.argtypes = [vp] * 9 + [I, I, I, I, F, I, I, vp, ctypes.c_size_t, I, vp]
        lib.fa_selftest_bwd_fault.restype = I
        lib.fa_fwd_kv_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.fa_fwd_kv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_kv.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, I, F, I, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_kv_splits_hint.argtypes = [I, I, I, I, I, I, I]
        lib.fa_fwd_kv_splits_hint.restype = I
        lib.fa_fwd_kv.restype = I
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, F, I, vp]
        lib.fa_fwd_fp8.restype = I
        lib.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, F, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_bwd.restype = I
        lib.fa_bwd_gqa.argtypes = [vp] * 9 + [I, I, I, I, I, F, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_bwd_gqa.restype = I
        lib.fa_fwd_host_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_host.restype = I
        lib.fa_bwd_host_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, F, I, I, vp, ctypes.c_size_t, vp]
        lib.fa_bwd_host.restype = I
        lib.fa_fwd_fp8_host_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_fwd_fp8_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_fwd_fp8_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, F, I, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_fp8_host.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def fa_fwd(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, D: int, scale: float,
           causal: int, dtype: int, stream: int) -> int:
    """Direct call of the C entry point; returns its status code."""
    return int(load_library().fa_fwd(q, k, v, o, lse, B, H, N, D, float(scale), int(causal), int(dtype),
                                     stream))


def fa_fwd_gqa(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, H_kv: int, N: int, D: int, scale: float,
               causal: int, dtype: int, stream: int) -> int:
    """Direct call of the grouped-K/V-head entry point; returns its status code."""
    return int(load_library().fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, D, float(scale), int(causal), int(dtype),
                                         stream))


def fa_splitkv_workspace_bytes(B: int, H: int, N: int, D: int, num_splits: int) -> int:
    return int(load_library().fa_splitkv_workspace_bytes(B, H, N, D, num_splits))


def fa_fwd_splitkv(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, D: int, scale: float,
                   causal: int, dtype: int, num_splits: int, workspace: int, workspace_bytes: int,
                   stream: int) -> int:
    """Direct call of the split-K entry point; returns its status code."""
    return int(load_library().fa_fwd_splitkv(q, k, v, o, lse, B, H, N, D, float(scale), int(causal), int(dtype),
                                             int(num_splits), workspace, int(workspace_bytes), stream))


def fa_fwd_splitkv_noalloc(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, D: int,
                           scale: float, causal: int, dtype: int, num_splits: int, stream: int) -> int:
    """Split-K forward for callers that cannot allocate device memory: the
    workspace is the library's fixed scratch buffer (see include/fa.h)."""
    return int(load_library().fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, N, D, float(scale), int(causal),
                                                     int(dtype), int(num_splits), stream))


def fa_noalloc_scratch_bytes() -> int:
    return int(load_library().fa_noalloc_scratch_bytes())


def fa_fwd_kv_workspace_bytes(B: int, H: int, Nq: int, D: int, num_splits: int) -> int:
    return int(load_library().fa_fwd_kv_workspace_bytes(B, H, Nq, D, num_splits))


def fa_fwd_kv(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, H_kv: int, Nq: int, Nk: int, D: int,
              scale: float, causal: int, dtype: int, num_splits: int, workspace: int, workspace_bytes: int,
              stream: int) -> int:
    """Direct call of the queries-against-a-K/V-sequence entry point; returns its status code."""
    return int(load_library().fa_fwd_kv(q, k, v, o, lse, B, H, H_kv, Nq, Nk, D, float(scale), int(causal),
                                        int(dtype), int(num_splits), workspace, int(workspace_bytes), stream))


def fa_fwd_kv_splits_hint(B: int, H: int, H_kv: int, Nq: int, Nk: int, D: int, causal: int) -> int:
    return int(load_library().fa_fwd_kv_splits_hint(B, H, H_kv, Nq, Nk, D, int(causal)))


def fa_fwd_fp8(q: int, k: int, v_t: int, q_scale: int, k_scale: int, v_scale: int, o: int, lse: int, B: int, H: int,
               N: int, D: int, scale: float, causal: int, stream: int) -> int:
    """Direct call of the FP8 (E4M3) forward entry point; returns its status code."""
    return int(load_library().fa_fwd_fp8(q, k, v_t, q_scale, k_scale, v_scale, o, lse, B, H, N, D, float(scale),
                                         int(causal), stream))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, D))


def fa_bwd(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int, H: int, N: int,
           D: int, scale: float, causal: int, dtype: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """Direct call of the backward entry point; returns its status code."""
    return int(load_library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, D, float(scale), int(causal),
                                     int(dtype), workspace, int(workspace_bytes), stream))


def fa_fwd_host_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(load_library().fa_fwd_host_workspace_bytes(B, H, N, D))


def fa_fwd_host(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, D: int, scale: float,
                causal: int, dtype: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """Direct call of the C entry point (q, k, v, o, lse: page-locked host pointers)."""
    return int(load_library().fa_fwd_host(q, k, v, o, lse, B, H, N, D, float(scale), int(causal), int(dtype),
                                          workspace, workspace_bytes, stream))


def fa_bwd_host_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(load_library().fa_bwd_host_workspace_bytes(B, H, N, D))


def fa_bwd_host(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int, H: int,
                N: int, D: int, scale: float, causal: int, dtype: int, workspace: int, workspace_bytes: int,
                stream: int) -> int:
    """Direct call of the C entry point (all tensors: page-locked host pointers)."""
    return int(load_library().fa_bwd_host(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, D, float(scale), int(causal),
                                          int(dtype), workspace, workspace_bytes, stream))


def fa_fwd_fp8_host_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(load_library().fa_fwd_fp8_host_workspace_bytes(B, H, N, D))


def fa_fwd_fp8_host(q: int, k: int, v_t: int, q_scale: int, k_scale: int, v_scale: int, o: int, lse: int, B: int,
                    H: int, N: int, D: int, scale: float, causal: int, workspace: int, workspace_bytes: int,
                    stream: int) -> int:
    """Direct call of the C entry point (all tensors: page-locked host pointers)."""
    return int(load_library().fa_fwd_fp8_host(q, k, v_t, q_scale, k_scale, v_scale, o, lse, B, H, N, D,
                                              float(scale), int(causal), workspace, workspace_bytes, stream))


def fa_bwd_gqa(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int, H: int,
               H_kv: int, N: int, D: int, scale: float, causal: int, dtype: int, workspace: int,
               workspace_bytes: int, stream: int) -> int:
    """Direct call of the C entry point; returns its status code."""
    return int(load_library().fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, D, float(scale),
                                         int(causal), int(dtype), workspace, workspace_bytes, stream))


def fa_get_device_status(stream: int) -> int:
    return int(load_library().fa_get_device_status(stream))


def fa_selftest_wait_timeout(stream: int) -> int:
    """Queue the bounded-wait self-test kernel (see include/fa.h)."""
    return int(load_library().fa_selftest_wait_timeout(stream))


def fa_selftest_fwd_fault(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, D: int, scale: float,
                          causal: int, dtype: int, fault_item: int, stream: int) -> int:
    """The forward kernel with one K/V copy left out (test of the give-up path;
    see include/fa.h)."""
    return int(load_library().fa_selftest_fwd_fault(q, k, v, o, lse, B, H, N, D, float(scale), int(causal),
                                                    int(dtype), int(fault_item), stream))


def fa_selftest_bwd_fault(q: int, k: int, v: int, o: int, dout: int, lse: int, dq: int, dk: int, dv: int, B: int,
                          H: int, N: int, D: int, scale: float, causal: int, dtype: int, workspace: int,
                          workspace_bytes: int, fault_step: int, stream: int) -> int:
    """The backward kernels with one Q copy left out (test of the give-up path;
    see include/fa.h)."""
    return int(load_library().fa_selftest_bwd_fault(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, D, float(scale),
                                                    int(causal), int(dtype), workspace, int(workspace_bytes),
                                                    int(fault_step), stream))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def attention(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
              num_splits: int = 0, workspace=None):
    """O, LSE = attention(Q, K, V) for contiguous fp16/bf16 CUDA tensors, Q [B,H,N,D]
    and K, V [B,H_kv,N,D] (H_kv = H, or a divisor of H for grouped K/V heads).

    Outputs are allocated with torch when not given.  Raises FaError on a
    non-OK status.  Asynchronous on ``stream`` (default: torch's current stream).
    ``num_splits`` > 0 selects the split-K path (fa_fwd_splitkv); its workspace
    is allocated with torch unless one is given.
    """
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or k.shape[0] != q.shape[0] or k.shape[2:] != q.shape[2:]:
        raise ValueError("q must be [B, H, N, D] and k, v [B, H_kv, N, D]")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("the query heads H must be a multiple of the K/V heads H_kv")
    H_kv = k.shape[1]
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    _same_device((q, k, v))
    B, H, N, D = q.shape
    _check_given(out, q.shape, q.dtype, "out", q.device)
    _check_given(lse, (B, H, N), torch.float32, "lse", q.device)
    _check_workspace(workspace, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    if num_splits > 0 and H_kv != H:
        raise ValueError("split-K with grouped K/V heads goes through attention_kv")
    if num_splits > 0:
        need = fa_splitkv_workspace_bytes(B, H, N, D, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, D,
                            scale, int(bool(causal)), dt, num_splits, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), handle)
        if st != FA_OK:
            raise FaError(st, "fa_fwd_splitkv")
        return out, lse
    if H_kv != H:
        st = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, H_kv, N, D,
                        scale, int(bool(causal)), dt, handle)
        if st != FA_OK:
            raise FaError(st, "fa_fwd_gqa")
        return out, lse
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, D, scale,
                int(bool(causal)), dt, handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return out, lse


def attention_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, workspace=None,
                   device=None, stream=None, synchronize: bool = True):
    """O, LSE = attention(Q, K, V) for contiguous fp16/bf16 tensors in PAGE-LOCKED
    host memory (``tensor.pin_memory()``), through fa_fwd_host: the copies to and
    from the GPU overlap the kernel.  Outputs are page-locked host tensors,
    allocated when not given; the device workspace is allocated with torch
    unless one is given.  With ``synchronize`` the call waits for the results;
    otherwise they are ready once ``stream`` has been synchronised.
    """
    import torch

    for t in (q, k, v):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("q, k, v must be page-locked host tensors")
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, H, N, D]")
    B, H, N, D = q.shape
    _check_given(out, q.shape, q.dtype, "out", pinned=True)
    _check_given(lse, (B, H, N), torch.float32, "lse", pinned=True)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check_workspace(workspace, device)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    need = fa_fwd_host_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    with torch.cuda.device(device):
        st = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, D,
                         scale, int(bool(causal)), dt, workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_host")
    if synchronize:
        stream.synchronize() if hasattr(stream, "synchronize") else torch.cuda.synchronize(device)
    return out, lse


def attention_backward_host(q, k, v, out, lse, dout, causal: bool = False, scale: float | None = None, dq=None,
                            dk=None, dv=None, workspace=None, device=None, stream=None, synchronize: bool = True):
    """dQ, dK, dV for contiguous fp16/bf16 tensors [B,H,N,D] (and the forward's
    fp32 LSE [B,H,N]) in PAGE-LOCKED host memory, through fa_bwd_host: the
    copies to and from the GPU overlap the kernels.  Gradients are page-locked
    host tensors, allocated when not given; the device workspace is allocated
    with torch unless one is given.  ``synchronize`` as for attention_host.
    """
    import torch

    for t in (q, k, v, out, dout, lse):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("q, k, v, out, dout and lse must be page-locked host tensors")
        if not t.is_contiguous():
            raise ValueError("q, k, v, out, dout and lse must be contiguous")
    if q.dtype not in (torch.float16, torch.bfloat16) or any(t.dtype != q.dtype for t in (k, v, out, dout)):
        raise ValueError("q, k, v, out, dout must share one dtype, float16 or bfloat16")
    if q.dim() != 4 or any(t.shape != q.shape for t in (k, v, out, dout)):
        raise ValueError("q, k, v, out, dout must all be [B, H, N, D]")
    B, H, N, D = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be float32 [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    for g, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_given(g, q.shape, q.dtype, name, pinned=True)
    _check_workspace(workspace, device)
    dq, dk, dv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) if g is None else g for g in (dq, dk, dv))
    need = fa_bwd_host_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    with torch.cuda.device(device):
        st = fa_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D, scale, int(bool(causal)), dt,
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_host")
    if synchronize:
        stream.synchronize() if hasattr(stream, "synchronize") else torch.cuda.synchronize(device)
    return dq, dk, dv


def attention_backward(q, k, v, out, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None,
                       dv=None, workspace=None, stream=None):
    """dQ, dK, dV of attention for contiguous fp16/bf16 CUDA tensors: q, out,
    dout [B,H,N,D] and k, v [B,H_kv,N,D] (H_kv = H, or a divisor of H for
    grouped K/V heads); ``out`` and ``lse`` are the forward pass's outputs,
    ``dout`` the upstream gradient.  Gradients (and the workspace) are
    allocated with torch when not given.  Raises FaError on a non-OK status.
    Asynchronous on ``stream``."""
    import torch

    ts = (q, k, v, out, dout)
    if not all(t.is_cuda for t in ts) or not lse.is_cuda:
        raise ValueError("all tensors must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16) or any(t.dtype != q.dtype for t in ts):
        raise ValueError("q, k, v, out, dout must share one dtype, float16 or bfloat16")
    if q.dim() != 4 or out.shape != q.shape or dout.shape != q.shape or k.dim() != 4 or v.shape != k.shape or \
            k.shape[0] != q.shape[0] or k.shape[2:] != q.shape[2:] or q.shape[1] % k.shape[1] != 0:
        raise ValueError("q, out, dout must be [B, H, N, D] and k, v [B, H_kv, N, D] with H_kv dividing H")
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be float32 [B, H, N]")
    if not all(t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("inputs must be contiguous")
    _same_device(ts + (lse,))
    _check_given(dq, q.shape, q.dtype, "dq", q.device)
    _check_given(dk, k.shape, q.dtype, "dk", q.device)
    _check_given(dv, k.shape, q.dtype, "dv", q.device)
    _check_workspace(workspace, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    need = fa_bwd_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    st = fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, N, D, scale, int(bool(causal)), dt,
                    workspace.data_ptr(), workspace.numel() * workspace.element_size(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_gqa")
    return dq, dk, dv


def attention_fp8(q8, k8, v8_t, q_scale, k_scale, v_scale, causal: bool = False, scale: float | None = None, out=None,
                  lse=None, stream=None):
    """O (bf16), LSE = attention of FP8 inputs: q8, k8 [B,H,N,D] and v8_t [B,H,D,N]
    (V transposed per head) as uint8 or float8_e4m3fn CUDA tensors, with fp32
    per-128-row block scales [B,H,ceil(N/128)].  Raises FaError on a non-OK
    status.  Asynchronous on ``stream``."""
    import torch

    ts = (q8, k8, v8_t)
    if not all(t.is_cuda and t.element_size() == 1 and t.is_contiguous() for t in ts):
        raise ValueError("q8, k8, v8_t must be contiguous 1-byte CUDA tensors")
    if q8.dim() != 4 or k8.shape != q8.shape:
        raise ValueError("q8, k8 must be [B, H, N, D]")
    B, H, N, D = q8.shape
    if tuple(v8_t.shape) != (B, H, D, N):
        raise ValueError("v8_t must be [B, H, D, N] (V transposed per head)")
    nb = (N + 127) // 128
    for t in (q_scale, k_scale, v_scale):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == (B, H, nb)):
            raise ValueError("scales must be contiguous float32 CUDA tensors [B, H, ceil(N/128)]")
    _same_device(ts + (q_scale, k_scale, v_scale))
    _check_given(out, (B, H, N, D), torch.bfloat16, "out", q8.device)
    _check_given(lse, (B, H, N), torch.float32, "lse", q8.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    if stream is None:
        stream = torch.cuda.current_stream(q8.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8_t.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                    v_scale.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, D, scale, int(bool(causal)), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return out, lse


def attention_kv(q, k, v, causal: bool = False, scale: float | None = None, num_splits=0, out=None, lse=None,
                 workspace=None, stream=None):
    """O, LSE for q [B,H,Nq,D] against k, v [B,H_kv,Nk,D] (fp16/bf16 CUDA tensors;
    query i is the token at position i + Nk - Nq).  ``num_splits`` > 0 selects
    split-K with a torch-allocated workspace unless one is given; "auto" takes
    fa_fwd_kv_splits_hint's choice."""
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3]:
        raise ValueError("q must be [B, H, Nq, D] and k, v [B, H_kv, Nk, D]")
    if not all(t.is_contiguous() for t in (q, k, v)):
        raise ValueError("q, k, v must be contiguous")
    _same_device((q, k, v))
    B, H, Nq, D = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    _check_given(out, q.shape, q.dtype, "out", q.device)
    _check_given(lse, (B, H, Nq), torch.float32, "lse", q.device)
    _check_workspace(workspace, q.device)
    if num_splits == "auto":
        with torch.cuda.device(q.device):
            num_splits = fa_fwd_kv_splits_hint(B, H, H_kv, Nq, Nk, D, int(bool(causal)))
        if num_splits < 0:
            raise FaError(1, "fa_fwd_kv_splits_hint")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_ptr, ws_bytes = 0, 0
    if num_splits > 0:
        need = fa_fwd_kv_workspace_bytes(B, H, Nq, D, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    dt = FA_BF16 if q.dtype == torch.bfloat16 else FA_FP16
    st = fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, H_kv, Nq, Nk, D,
                   scale, int(bool(causal)), dt, num_splits, ws_ptr, ws_bytes, handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_kv")
    return out, lse
