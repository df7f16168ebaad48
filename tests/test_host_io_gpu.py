"""fa_fwd_host and fa_bwd_host (tensors in page-locked host memory, copies
overlapped with the kernels in chunks of (b, h) planes), through the C ABI.

Every plane is computed by the device kernels, so the forward results must
equal fa_fwd's bit for bit, and dK, dV fa_bwd's (dQ is summed with fp32
atomics in both, so only the order of its additions differs); small cases are
also checked against the FP64 oracle with the device paths' tolerances.  The
shapes cover one chunk, several chunks, chunk boundaries that must be moved to
keep the LSE rows 16-byte aligned (odd and even N), and both dtypes.
"""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu


def _pinned(w, seed):
    return [t.pin_memory() for t in fa_inputs.make_qkv(w, seed=seed)]


@pytest.mark.parametrize("B,H,N,D,causal,dtype", [
    (1, 2, 256, 64, False, "fp16"),      # one chunk
    (2, 3, 333, 128, True, "bf16"),      # one chunk, odd N
    (1, 32, 4097, 64, True, "fp16"),     # four chunks of 8 planes (N odd: a multiple of 4 planes)
    (2, 16, 4096, 64, True, "fp16"),     # four chunks
    (1, 24, 8190, 64, False, "bf16"),    # N = 2 mod 4: six chunks of an even number of planes
    (1, 32, 8192, 128, True, "fp16"),    # the bench workload: eight chunks
])
def test_equals_device_path(B, H, N, D, causal, dtype):
    w = fa_inputs.Workload("host", B, H, N, D, causal, dtype)
    q, k, v = _pinned(w, seed=N + H)
    o, lse = fa.attention_host(q, k, v, causal=causal, scale=w.scale)
    assert fa.fa_get_device_status(0) == fa.FA_OK
    od, ld = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert not o.is_cuda and o.is_pinned()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_against_oracle():
    w = fa_inputs.WORKLOADS["tiny_fp16_b1h2n256d64"].with_(causal=True)
    q, k, v = _pinned(w, seed=0)
    o, lse = fa.attention_host(q, k, v, causal=True, scale=w.scale)
    o_ref, lse_ref = fa_ref.naive(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), w.scale, True,
                                  enc=fa_inputs.enc(w))
    assert float(np.abs(o.float().numpy() - o_ref).max()) <= 2e-3
    assert float(np.abs(lse.numpy() - lse_ref).max()) <= 1e-3


def test_stream_order_and_workspace_reuse():
    """Two calls queued back to back on one side stream with one workspace:
    the second call's copies wait for the first call's, and the stream is
    ordered after the copies back."""
    w = fa_inputs.Workload("host2", 1, 16, 1024, 128, True, "fp16")
    a = _pinned(w, seed=1)
    b = _pinned(w, seed=2)
    ws = torch.empty(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.D), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    oa, la = fa.attention_host(*a, causal=True, workspace=ws, stream=s, synchronize=False)
    ob, lb = fa.attention_host(*b, causal=True, workspace=ws, stream=s, synchronize=False)
    s.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    for (q, k, v), o, lse in ((a, oa, la), (b, ob, lb)):
        od, ld = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_argument_errors_queue_nothing():
    w = fa_inputs.Workload("host3", 1, 2, 256, 64, False, "fp16")
    q, k, v = _pinned(w, seed=3)
    o = torch.full(q.shape, 7.0, dtype=q.dtype).pin_memory()
    lse = torch.full((1, 2, 256), 7.0).pin_memory()
    need = fa.fa_fwd_host_workspace_bytes(1, 2, 256, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(q.shape, dtype=q.dtype)
    host_ws = torch.empty(need, dtype=torch.uint8).pin_memory()
    call = lambda qq, oo, wsp, wsb, D=64: fa.fa_fwd_host(qq.data_ptr(), k.data_ptr(), v.data_ptr(), oo.data_ptr(),
                                                        lse.data_ptr(), 1, 2, 256, D, w.scale, 0, fa.FA_FP16,
                                                        wsp, wsb, 0)
    assert call(pageable, o, ws.data_ptr(), need) == 1            # input not page-locked
    assert call(q, pageable, ws.data_ptr(), need) == 1            # output not page-locked
    assert call(q, o, host_ws.data_ptr(), need) == 1              # workspace not device memory
    assert call(q, o, ws.data_ptr(), need - 256) == 1             # workspace too small
    assert call(q, o, ws.data_ptr() + 16, need - 256) == 3        # workspace not 256-byte aligned
    assert call(q, o, ws.data_ptr(), need, D=96) == 2
    torch.cuda.synchronize()
    assert (o == 7).all() and (lse == 7).all()
    assert fa.fa_get_device_status(0) == fa.FA_OK


# ------------------------------------------------------------------ fa_bwd_host

def _bwd_pinned(w, seed):
    q, k, v = fa_inputs.make_qkv(w, seed=seed)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(seed + 1)).to(q.dtype)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    return [t.pin_memory() for t in (q, k, v, o.cpu(), do, lse.cpu())]


@pytest.mark.parametrize("B,H,N,D,causal,dtype", [
    (1, 2, 256, 64, True, "fp16"),       # one chunk
    (2, 3, 333, 128, False, "bf16"),     # one chunk, odd N
    (1, 16, 4097, 64, True, "fp16"),     # four chunks of 4 planes (N odd)
    (1, 32, 8192, 128, True, "fp16"),    # the bench workload: eight chunks
])
def test_backward_equals_device_path(B, H, N, D, causal, dtype):
    w = fa_inputs.Workload("bwdhost", B, H, N, D, causal, dtype)
    q, k, v, o, do, lse = _bwd_pinned(w, seed=N + D)
    dq, dk, dv = fa.attention_backward_host(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    assert fa.fa_get_device_status(0) == fa.FA_OK
    assert not dq.is_cuda and dq.is_pinned()
    rq, rk, rv = fa.attention_backward(*(t.cuda() for t in (q, k, v, o, lse, do)), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dk, rk.cpu()) and torch.equal(dv, rv.cpu())
    # dQ: fp32 atomics in both, so only the order of the additions differs
    tol = 2.0 ** -9 * max(1.0, rq.float().abs().max().item())
    assert (dq.float() - rq.cpu().float()).abs().max().item() <= tol


def test_backward_against_oracle():
    w = fa_inputs.WORKLOADS["tiny_fp16_b1h2n256d64"].with_(causal=True)
    q, k, v, o, do, lse = _bwd_pinned(w, seed=5)
    dq, dk, dv = fa.attention_backward_host(q, k, v, o, lse, do, causal=True, scale=w.scale)
    refs = fa_ref.backward(*(fa_inputs.bits(t) for t in (q, k, v, do)), w.scale, True, enc=fa_inputs.enc(w))
    for got, ref in zip((dq, dk, dv), refs):
        assert float(np.abs(got.float().numpy() - ref).max()) <= 2.0 ** -9 * max(1.0, float(np.abs(ref).max()))


def test_backward_argument_errors_queue_nothing():
    w = fa_inputs.Workload("bwdhost3", 1, 2, 256, 64, False, "fp16")
    q, k, v, o, do, lse = _bwd_pinned(w, seed=9)
    dq, dk, dv = (torch.full(q.shape, 7.0, dtype=q.dtype).pin_memory() for _ in range(3))
    need = fa.fa_bwd_host_workspace_bytes(1, 2, 256, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(q.shape, dtype=q.dtype)
    call = lambda dout, g, wsb: fa.fa_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                               dout.data_ptr(), lse.data_ptr(), g.data_ptr(), dk.data_ptr(),
                                               dv.data_ptr(), 1, 2, 256, 64, w.scale, 0, fa.FA_FP16, ws.data_ptr(),
                                               wsb, 0)
    assert call(pageable, dq, need) == 1          # dO not page-locked
    assert call(do, pageable, need) == 1          # dQ not page-locked
    assert call(do, dq, need - 256) == 1          # workspace too small
    torch.cuda.synchronize()
    assert all((g == 7).all() for g in (dq, dk, dv))
    assert fa.fa_get_device_status(0) == fa.FA_OK


# ------------------------------------------------------------------ fa_fwd_fp8_host

@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 256, False), (2, 3, 400, True), (1, 32, 4096, True)])
def test_fp8_equals_device_path(B, H, N, causal):
    w = fa_inputs.Workload("fp8host", B, H, N, 128, causal, "bf16")
    (q8, k8, v8), scs = fa_inputs.make_qkv_fp8(w, seed=N)
    vt = v8.transpose(2, 3).contiguous()
    hq, hk, hv = (t.pin_memory() for t in (q8, k8, vt))
    hs = [t.pin_memory() for t in scs]
    o = torch.empty((B, H, N, 128), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, N)).pin_memory()
    nb = fa.fa_fwd_fp8_host_workspace_bytes(B, H, N, 128)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = fa.fa_fwd_fp8_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), *(t.data_ptr() for t in hs), o.data_ptr(),
                            lse.data_ptr(), B, H, N, 128, w.scale, int(causal), ws.data_ptr(), nb, 0)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    od, ld = fa.attention_fp8(q8.cuda(), k8.cuda(), vt.cuda(), *(t.cuda() for t in scs), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
