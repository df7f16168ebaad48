"""ctypes wrapper of the FP64 CPU oracle (``oracle/fa_ref.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The CUDA path neither
imports this module nor links the library, and this module imports nothing
from the CUDA path.

Inputs are numpy arrays shaped [B, H, N, D] (or [N, D], read as B = H = 1):
  * float64 arrays are used as they are (``enc="f64"``);
  * 16-bit inputs are passed as their raw bit patterns in a uint16 array with
    ``enc="f16"`` (IEEE binary16) or ``enc="bf16"`` (bfloat16); the oracle
    decodes them exactly to double before any arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_ref.c")
_HDR = os.path.join(_HERE, "fa_ref.h")
_LIB = os.path.join(_HERE, "libfa_ref.so")

ENC = {"f64": 0, "f16": 1, "bf16": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) if it is stale."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, dp, lp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_long)
        L, I, Dbl = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.fa_ref_naive.argtypes = [vp, vp, vp, I, dp, dp, L, L, L, L, Dbl, I, I]
        lib.fa_ref_naive.restype = I
        lib.fa_ref_naive_rows.argtypes = [vp, vp, vp, I, L, L, L, L, Dbl, I, lp, lp, L, dp, dp, I]
        lib.fa_ref_naive_rows.restype = I
        lib.fa_ref_blocked.argtypes = [vp, vp, vp, I, dp, dp, L, L, L, L, Dbl, I, L, L, I, I,
                                       L, dp, L, lp, lp, I]
        lib.fa_ref_blocked.restype = I
        lib.fa_ref_split_merge.argtypes = [vp, vp, vp, I, dp, dp, L, L, L, L, Dbl, I, L, dp, dp, L, I]
        lib.fa_ref_split_merge.restype = I
        lib.fa_ref_naive_gqa.argtypes = [vp, vp, vp, I, dp, dp, L, L, L, L, L, Dbl, I, I]
        lib.fa_ref_naive_gqa.restype = I
        lib.fa_ref_backward.argtypes = [vp, vp, vp, vp, I, dp, dp, dp, dp, L, L, L, L, Dbl, I, I]
        lib.fa_ref_backward.restype = I
        lib.fa_ref_backward_sample.argtypes = [vp, vp, vp, vp, I, L, L, L, L, Dbl, I, lp, lp, L, dp,
                                               lp, lp, L, dp, dp, I]
        lib.fa_ref_backward_sample.restype = I
        lib.fa_ref_naive_kv.argtypes = [vp, vp, vp, I, dp, dp, L, L, L, L, L, L, Dbl, I, I]
        lib.fa_ref_naive_kv.restype = I
        lib.fa_ref_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.fa_ref_decode_e4m3.restype = Dbl
        lib.fa_ref_dequant_e4m3.argtypes = [vp, ctypes.POINTER(ctypes.c_float), L, L, L, L, dp]
        lib.fa_ref_dequant_e4m3.restype = I
        lib.fa_ref_max_threads.argtypes = []
        lib.fa_ref_max_threads.restype = I
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().fa_ref_max_threads())


def _prep(q, k, v, enc):
    if enc not in ENC:
        raise ValueError("enc must be one of %s" % sorted(ENC))
    want = np.float64 if enc == "f64" else np.uint16
    arrs = []
    for t in (q, k, v):
        a = np.ascontiguousarray(t)
        if a.dtype != want:
            raise TypeError("enc=%s needs %s arrays, got %s" % (enc, np.dtype(want), a.dtype))
        if a.ndim == 2:
            a = a.reshape(1, 1, *a.shape)
        if a.ndim != 4:
            raise ValueError("inputs must be [B,H,N,D] or [N,D]")
        arrs.append(a)
    if not (arrs[0].shape == arrs[1].shape == arrs[2].shape):
        raise ValueError("q, k, v shapes differ")
    return arrs


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def naive(q, k, v, scale, causal=False, enc="f64", nthreads=0):
    """Safe-softmax attention of every row; returns (O [B,H,N,D], LSE [B,H,N])."""
    q, k, v = _prep(q, k, v, enc)
    B, H, N, D = q.shape
    o = np.empty((B, H, N, D), np.float64)
    lse = np.empty((B, H, N), np.float64)
    rc = _load().fa_ref_naive(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc],
                              _dptr(o), _dptr(lse), B, H, N, D, float(scale), int(bool(causal)),
                              int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_naive failed (%d)" % rc)
    return o, lse


def naive_rows(q, k, v, scale, causal, bh_idx, row_idx, enc="f64", nthreads=0):
    """Safe-softmax attention of selected rows: returns (O [R,D], LSE [R])."""
    q, k, v = _prep(q, k, v, enc)
    B, H, N, D = q.shape
    bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
    rows = np.ascontiguousarray(row_idx, dtype=np.int64)
    if bh.shape != rows.shape or bh.ndim != 1:
        raise ValueError("bh_idx and row_idx must be 1-D and of equal length")
    R = bh.shape[0]
    o = np.empty((R, D), np.float64)
    lse = np.empty((R,), np.float64)
    lp = ctypes.POINTER(ctypes.c_long)
    rc = _load().fa_ref_naive_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc],
                                   B, H, N, D, float(scale), int(bool(causal)),
                                   bh.ctypes.data_as(lp), rows.ctypes.data_as(lp), R,
                                   _dptr(o), _dptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_naive_rows failed (%d)" % rc)
    return o, lse


def blocked(q, k, v, scale, causal=False, Br=64, Bc=64, kv_outer=False, rescale=True,
            trace_row=None, trace_cap=4096, enc="f64", nthreads=0):
    """Blocked online-softmax attention.

    Returns (O, LSE, trace, visited): ``trace`` is an array of rows
    (j0, m_new, l_new, corr) for query row ``trace_row`` of head 0 (None when
    no row is traced); ``visited`` is the number of block pairs computed for
    one head.
    """
    q, k, v = _prep(q, k, v, enc)
    B, H, N, D = q.shape
    o = np.empty((B, H, N, D), np.float64)
    lse = np.empty((B, H, N), np.float64)
    tr = np.zeros((trace_cap, 4), np.float64) if trace_row is not None else None
    tlen = ctypes.c_long(0)
    vis = ctypes.c_long(0)
    rc = _load().fa_ref_blocked(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc],
                                _dptr(o), _dptr(lse), B, H, N, D, float(scale),
                                int(bool(causal)), int(Br), int(Bc), int(bool(kv_outer)),
                                int(bool(rescale)),
                                -1 if trace_row is None else int(trace_row),
                                _dptr(tr) if tr is not None else None,
                                trace_cap if tr is not None else 0,
                                ctypes.byref(tlen), ctypes.byref(vis), int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_blocked failed (%d)" % rc)
    return o, lse, (tr[: tlen.value].copy() if tr is not None else None), int(vis.value)


def split_merge(q, k, v, scale, causal=False, chunk=128, enc="f64", nthreads=0, parts=0):
    """Keys cut into chunks of `chunk`, partial (m, l, o) per chunk, merged.

    Returns (O, LSE) or, with parts > 0, (O, LSE, m_parts, l_parts) where the
    partials are those of row 0 of head 0.
    """
    q, k, v = _prep(q, k, v, enc)
    B, H, N, D = q.shape
    o = np.empty((B, H, N, D), np.float64)
    lse = np.empty((B, H, N), np.float64)
    pm = np.zeros(max(parts, 1), np.float64)
    pl = np.zeros(max(parts, 1), np.float64)
    rc = _load().fa_ref_split_merge(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc], _dptr(o), _dptr(lse),
                                    B, H, N, D, float(scale), int(bool(causal)), int(chunk),
                                    _dptr(pm) if parts else None, _dptr(pl) if parts else None, int(parts),
                                    int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_split_merge failed (%d)" % rc)
    return (o, lse, pm[:parts], pl[:parts]) if parts else (o, lse)


def naive_gqa(q, k, v, scale, causal=False, enc="f64", nthreads=0):
    """Safe-softmax attention with grouped K/V heads: q [B,H,N,D], k/v
    [B,H_kv,N,D]; returns (O [B,H,N,D], LSE [B,H,N])."""
    want = np.float64 if enc == "f64" else np.uint16
    q, k, v = (np.ascontiguousarray(t) for t in (q, k, v))
    for t in (q, k, v):
        if t.dtype != want or t.ndim != 4:
            raise TypeError("enc=%s needs 4-D %s arrays" % (enc, np.dtype(want)))
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, D) or v.shape != k.shape:
        raise ValueError("k, v must be [B, H_kv, N, D]")
    o = np.empty((B, H, N, D), np.float64)
    lse = np.empty((B, H, N), np.float64)
    rc = _load().fa_ref_naive_gqa(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc], _dptr(o), _dptr(lse),
                                  B, H, H_kv, N, D, float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_naive_gqa failed (%d)" % rc)
    return o, lse


def backward(q, k, v, dout, scale, causal=False, enc="f64", nthreads=0):
    """Gradients of attention for the upstream gradient dout = dL/dO.

    Returns (dQ, dK, dV, Delta): dQ, dK, dV [B,H,N,D] and Delta [B,H,N]
    (Delta_i = rowsum(dP_i * P_i)), all float64."""
    q, k, v = _prep(q, k, v, enc)
    (g,) = _prep_like(dout, q, enc)
    B, H, N, D = q.shape
    dq = np.empty((B, H, N, D), np.float64)
    dk = np.empty((B, H, N, D), np.float64)
    dv = np.empty((B, H, N, D), np.float64)
    delta = np.empty((B, H, N), np.float64)
    rc = _load().fa_ref_backward(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, ENC[enc],
                                 _dptr(dq), _dptr(dk), _dptr(dv), _dptr(delta), B, H, N, D, float(scale),
                                 int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_backward failed (%d)" % rc)
    return dq, dk, dv, delta


def backward_sample(q, k, v, dout, scale, causal, dq_bh, dq_rows, kv_bh, kv_keys, enc="f64", nthreads=0):
    """Selected gradient rows: returns (dQ [R,D] of (dq_bh[r], dq_rows[r]),
    dK [S,D] and dV [S,D] of (kv_bh[s], kv_keys[s]))."""
    q, k, v = _prep(q, k, v, enc)
    (g,) = _prep_like(dout, q, enc)
    B, H, N, D = q.shape
    lp = ctypes.POINTER(ctypes.c_long)
    a_bh, a_rows, b_bh, b_keys = (np.ascontiguousarray(x, dtype=np.int64) for x in (dq_bh, dq_rows, kv_bh, kv_keys))
    if a_bh.shape != a_rows.shape or b_bh.shape != b_keys.shape:
        raise ValueError("index arrays of a pair must have the same length")
    R, S = a_bh.shape[0], b_bh.shape[0]
    dq = np.empty((max(R, 1), D), np.float64)
    dk = np.empty((max(S, 1), D), np.float64)
    dv = np.empty((max(S, 1), D), np.float64)
    rc = _load().fa_ref_backward_sample(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, ENC[enc],
                                        B, H, N, D, float(scale), int(bool(causal)),
                                        a_bh.ctypes.data_as(lp), a_rows.ctypes.data_as(lp), R, _dptr(dq),
                                        b_bh.ctypes.data_as(lp), b_keys.ctypes.data_as(lp), S, _dptr(dk), _dptr(dv),
                                        int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_backward_sample failed (%d)" % rc)
    return dq[:R], dk[:S], dv[:S]


def _prep_like(t, ref, enc):
    want = np.float64 if enc == "f64" else np.uint16
    a = np.ascontiguousarray(t)
    if a.dtype != want:
        raise TypeError("enc=%s needs %s arrays, got %s" % (enc, np.dtype(want), a.dtype))
    if a.ndim == 2:
        a = a.reshape(1, 1, *a.shape)
    if a.shape != ref.shape:
        raise ValueError("dout must have the shape of q")
    return (a,)


def decode_e4m3(byte):
    """Exact value of one OCP E4M3 byte (NaN for the NaN patterns)."""
    return float(_load().fa_ref_decode_e4m3(int(byte) & 0xff))


def dequant_e4m3(x_bytes, block_scale, block_rows=128):
    """x_bytes [B,H,N,D] uint8 (E4M3 bit patterns), block_scale [B,H,ceil(N/block_rows)]
    float32 -> float64 [B,H,N,D] = decode(x) * scale of the row's block."""
    x = np.ascontiguousarray(x_bytes, dtype=np.uint8)
    if x.ndim != 4:
        raise ValueError("x must be [B, H, N, D]")
    B, H, N, D = x.shape
    nb = (N + block_rows - 1) // block_rows
    sc = np.ascontiguousarray(block_scale, dtype=np.float32)
    if sc.shape != (B, H, nb):
        raise ValueError("block_scale must be [B, H, %d]" % nb)
    out = np.empty((B, H, N, D), np.float64)
    rc = _load().fa_ref_dequant_e4m3(x.ctypes.data, sc.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), B * H, N, D,
                                     block_rows, _dptr(out))
    if rc != 0:
        raise RuntimeError("fa_ref_dequant_e4m3 failed (%d)" % rc)
    return out


def naive_kv(q, k, v, scale, causal=False, enc="f64", nthreads=0):
    """q [B,H,Nq,D] against k, v [B,H_kv,Nk,D] (Nk >= Nq when causal; query i is
    sequence position i + Nk - Nq).  Returns (O [B,H,Nq,D], LSE [B,H,Nq])."""
    want = np.float64 if enc == "f64" else np.uint16
    q, k, v = (np.ascontiguousarray(t) for t in (q, k, v))
    for t in (q, k, v):
        if t.dtype != want or t.ndim != 4:
            raise TypeError("enc=%s needs 4-D %s arrays" % (enc, np.dtype(want)))
    B, H, Nq, D = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, H_kv, Nk, D) or v.shape != k.shape:
        raise ValueError("k, v must be [B, H_kv, Nk, D]")
    o = np.empty((B, H, Nq, D), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = _load().fa_ref_naive_kv(q.ctypes.data, k.ctypes.data, v.ctypes.data, ENC[enc], _dptr(o), _dptr(lse),
                                 B, H, H_kv, Nq, Nk, D, float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError("fa_ref_naive_kv failed (%d)" % rc)
    return o, lse
