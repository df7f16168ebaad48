"""The give-up path of the real forward and backward kernels.

The FlashAttention-on-MI50 engineering page (kwkr.cn, section 3.1, its fault
tree) lists a timing violation among the causes of a kernel that never
finishes.  Here every mbarrier wait is bounded instead: a role that waits
longer than 1 s records a status bit, raises the CTA's abort flag so that the
other roles stop waiting, lets the copies and UMMAs it issued finish, and the
CTA frees its tensor memory and returns.

fa_selftest_fwd_fault / fa_selftest_bwd_fault launch the same kernels as
fa_fwd / fa_bwd with one load left out on purpose (the K/V producer skips one
ring item; the backward loader skips one Q tile), so that path runs in the
kernels themselves.  Each test checks that the launch is reported as
FA_ERR_TIMEOUT within a few seconds, that reading the status clears it, and
that the next ordinary call on the same context matches the FP64 oracle.
Nothing here faults, traps or hangs the GPU: the only failure is a wait that
runs out.
"""
import time

import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 5


def _dt(w):
    return fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP16


def _forward_matches_oracle(w, seed):
    q, k, v = fa_inputs.make_qkv(w, seed=seed)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    o_ref, lse_ref = fa_ref.naive(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), w.scale, w.causal,
                                  enc=fa_inputs.enc(w))
    tol = 2e-3 if w.dtype == "fp16" else 1e-2
    assert float(np.abs(o.float().cpu().numpy() - o_ref).max()) <= tol
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= 1e-3


# The first two problems have fewer 256-row work tiles than SMs, so they run in
# the key-split form (ring items of a work tile: K, V of stream 0's first K/V
# tile, K, V of stream 1's first, then the second ones, ...); the third runs in
# the 256-row form (K_0, V_0, K_1, V_1, ... shared by both streams).
@pytest.mark.parametrize("B,H,N,D,causal,item", [
    (1, 2, 1000, 64, True, 5),       # V of stream 0's second K/V tile, P V of earlier steps in flight
    (1, 2, 300, 128, False, 0),      # stream 0's first K: nothing issued yet when the wait runs out
    (1, 32, 2048, 128, True, 21),    # V_10 of the first work tile of some CTAs, V_0 or V_2 of the second of others
])
def test_forward_gives_up_and_context_survives(B, H, N, D, causal, item):
    w = fa_inputs.Workload("fault", B, H, N, D, causal, "fp16")
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=21))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    s = torch.cuda.Stream()
    t0 = time.time()
    st = fa.fa_selftest_fwd_fault(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                  D, w.scale, int(causal), _dt(w), item, s.cuda_stream)
    assert st == fa.FA_OK
    assert fa.fa_get_device_status(s.cuda_stream) == FA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert fa.fa_get_device_status(s.cuda_stream) == fa.FA_OK   # reading clears it
    _forward_matches_oracle(fa_inputs.Workload("after", 1, 2, 700, D, causal, "fp16"), seed=22)


@pytest.mark.parametrize("N,D,causal,step", [
    (1000, 64, True, 3),     # a Q tile in the middle of the first work tile
    (700, 128, False, 0),    # the first Q tile: nothing issued yet
])
def test_backward_gives_up_and_context_survives(N, D, causal, step):
    w = fa_inputs.Workload("bfault", 1, 2, N, D, causal, "bf16")
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=31))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(32)).to(q.dtype).cuda()
    o, lse = fa.attention(q, k, v, causal=causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws_bytes = fa.fa_bwd_workspace_bytes(1, 2, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    s = torch.cuda.Stream()
    t0 = time.time()
    st = fa.fa_selftest_bwd_fault(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                  lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, 2, N, D, w.scale,
                                  int(causal), _dt(w), ws.data_ptr(), ws_bytes, step, s.cuda_stream)
    assert st == fa.FA_OK
    assert fa.fa_get_device_status(s.cuda_stream) == FA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert fa.fa_get_device_status(s.cuda_stream) == fa.FA_OK
    # the ordinary backward pass on the same context and inputs
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    refs = fa_ref.backward(*(fa_inputs.bits(t.cpu()) for t in (q, k, v, do)), w.scale, causal,
                           enc=fa_inputs.enc(w))
    for got, ref in zip((dq, dk, dv), refs):
        tol = 2.0 ** -6 * max(1.0, float(np.abs(ref).max()))
        assert float(np.abs(got.float().cpu().numpy() - ref).max()) <= tol


def test_fault_index_must_be_non_negative():
    w = fa_inputs.Workload("fneg", 1, 1, 128, 64, False, "fp16")
    q = torch.zeros(1, 1, 128, 64, device="cuda", dtype=torch.float16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 128, device="cuda")
    assert fa.fa_selftest_fwd_fault(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1,
                                    128, 64, w.scale, 0, fa.FA_FP16, -1, 0) == 1
