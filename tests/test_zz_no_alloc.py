"""fa_fwd_splitkv_noalloc: the split-K forward pass for callers that cannot
allocate device memory (a framework that owns all device memory, or a loop
where cudaMalloc / cudaFree and their device-wide synchronisation are not
allowed).  Its scratch is a fixed buffer inside the library, so it is checked
against the entry point that takes a caller workspace, on two calls in a row
with different inputs (the shared buffer keeps the previous call's contents,
and that must not leak into the next result)."""
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs

pytestmark = pytest.mark.gpu


def _split_with_workspace(q, k, v, causal, scale, splits):
    B, H, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=q.device)
    need = fa.fa_splitkv_workspace_bytes(B, H, N, D, splits)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    dt = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_FP16
    st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D,
                           scale, int(causal), dt, splits, ws.data_ptr(), need, 0)
    assert st == fa.FA_OK
    return o, lse


def _split_no_alloc(q, k, v, causal, scale, splits):
    B, H, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=q.device)
    dt = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_FP16
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                   N, D, scale, int(causal), dt, splits, 0)
    assert st == fa.FA_OK
    return o, lse


def test_no_alloc_matches_workspace_entry_on_two_calls():
    cases = [fa_inputs.Workload("na1", 1, 4, 1000, 128, True, "fp16"),
             fa_inputs.Workload("na2", 2, 3, 777, 64, False, "bf16")]
    tol = {"fp16": 2e-3, "bf16": 1e-2}
    for call, (w, splits) in enumerate(zip(cases, (4, 3))):
        assert fa.fa_splitkv_workspace_bytes(w.B, w.H, w.N, w.D, splits) <= fa.fa_noalloc_scratch_bytes()
        q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=10 + call))
        o_ref, lse_ref = _split_with_workspace(q, k, v, w.causal, w.scale, splits)
        o, lse = _split_no_alloc(q, k, v, w.causal, w.scale, splits)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(0) == fa.FA_OK
        assert (o.float() - o_ref.float()).abs().max().item() <= tol[w.dtype], "call %d" % call
        assert (lse - lse_ref).abs().max().item() <= 1e-3, "call %d" % call


def test_no_alloc_rejects_problems_beyond_its_scratch():
    # 64 splits of B1 H32 N4096 D128 need 64 * 131072 * 528 bytes, far over 64 MiB
    B, H, N, D, S = 1, 32, 4096, 128, 64
    assert fa.fa_splitkv_workspace_bytes(B, H, N, D, S) > fa.fa_noalloc_scratch_bytes()
    q = torch.zeros(B, H, N, D, device="cuda", dtype=torch.float16)
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, N), 3.0, device="cuda")
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                   D, 0.1, 1, fa.FA_FP16, S, 0)
    assert st == 6 and fa.fa_status_string(st) == "FA_ERR_TOO_LARGE"
    torch.cuda.synchronize()
    assert (o == 3).all() and (lse == 3).all()
