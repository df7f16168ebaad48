"""fa_fwd_splitkv_noalloc: the split-K forward pass for callers that cannot
allocate device memory.  Such callers are, for example, a framework that owns
every device allocation and hands the library only its tensors, or a loop in
which cudaMalloc / cudaFree are not allowed because they can synchronise the
whole device.  The entry point's scratch is a fixed buffer inside the library,
shared by every call on a device, which keeps the previous call's contents.

The checks, through the C ABI, on two calls in a row:
  * each call gives exactly (bit for bit) what fa_fwd_splitkv gives with a
    caller workspace on the same inputs: both run the same kernels, so any
    difference would be stale scratch leaking into a result;
  * the first call is a large non-causal one that fills the whole region the
    second call uses with non-zero partials; the second is causal with split
    chunks that hold no visible key, whose (m, l) = (-inf, 0) must be written,
    not inherited;
  * the second call also matches the FP64 oracle within the parity tolerance.
This file is collected last, so a run that stops at the first failure has run
every other test before it.
"""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu


def _dt(q):
    return fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_FP16


def _split_with_workspace(q, k, v, causal, scale, splits):
    B, H, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=q.device)
    need = fa.fa_splitkv_workspace_bytes(B, H, N, D, splits)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D,
                           scale, int(causal), _dt(q), splits, ws.data_ptr(), need, 0)
    assert st == fa.FA_OK
    return o, lse


def _split_no_alloc(q, k, v, causal, scale, splits):
    B, H, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=q.device)
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                   N, D, scale, int(causal), _dt(q), splits, 0)
    assert st == fa.FA_OK
    return o, lse


def test_no_alloc_matches_workspace_entry_on_two_calls():
    # call 0: 4 * 8 * 2048 * 128 * 4 bytes = 32 MiB of partial O, all non-zero, at
    # the start of the scratch; call 1 needs 4 * 4 * 1000 * 528 bytes = 8.4 MB
    # of it.  In call 1 (N = 1000, 4 splits) the first query block sees 2 K/V
    # tiles, so its chunks 2 and 3 hold no key.
    cases = [(fa_inputs.Workload("na0", 1, 8, 2048, 128, False, "fp16"), 4),
             (fa_inputs.Workload("na1", 1, 4, 1000, 128, True, "fp16"), 4)]
    first = fa.fa_splitkv_workspace_bytes(1, 8, 2048, 128, 4) - 4 * 8 * 2048 * 16
    assert fa.fa_splitkv_workspace_bytes(1, 4, 1000, 128, 4) <= first
    for call, (w, splits) in enumerate(cases):
        assert fa.fa_splitkv_workspace_bytes(w.B, w.H, w.N, w.D, splits) <= fa.fa_noalloc_scratch_bytes()
        q_h, k_h, v_h = fa_inputs.make_qkv(w, seed=10 + call)
        q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
        o, lse = _split_no_alloc(q, k, v, w.causal, w.scale, splits)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(0) == fa.FA_OK
        o_ws, lse_ws = _split_with_workspace(q, k, v, w.causal, w.scale, splits)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(0) == fa.FA_OK
        assert torch.equal(o, o_ws), "call %d: O differs from fa_fwd_splitkv" % call
        assert torch.equal(lse, lse_ws), "call %d: LSE differs from fa_fwd_splitkv" % call
        if call == 1:
            o_ref, lse_ref = fa_ref.naive(fa_inputs.bits(q_h), fa_inputs.bits(k_h), fa_inputs.bits(v_h), w.scale,
                                          w.causal, enc=fa_inputs.enc(w))
            assert float(np.abs(o.float().cpu().numpy() - o_ref).max()) <= 2e-3
            assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= 1e-3


def test_no_alloc_rejects_problems_beyond_its_scratch():
    # 64 splits of B1 H32 N4096 D128 need 64 * 131072 * 528 bytes, far over 64 MiB
    B, H, N, D, S = 1, 32, 4096, 128, 64
    assert fa.fa_splitkv_workspace_bytes(B, H, N, D, S) > fa.fa_noalloc_scratch_bytes()
    q = torch.zeros(B, H, N, D, device="cuda", dtype=torch.float16)
    k, v = torch.zeros_like(q), torch.zeros_like(q)
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, N), 3.0, device="cuda")
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                   D, 0.1, 1, fa.FA_FP16, S, 0)
    assert st == 6 and fa.fa_status_string(st) == "FA_ERR_TOO_LARGE"
    torch.cuda.synchronize()
    assert (o == 3).all() and (lse == 3).all()
