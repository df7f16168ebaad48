"""The torch wrappers reject caller-provided outputs and workspaces that do not
match what the kernels write (shape, dtype, contiguity, device or page-locked
host memory) before anything is launched: the C ABI sees only pointers, so a
short output would otherwise be written past its end.  Correct ones are used."""
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs

pytestmark = pytest.mark.gpu


def _qkv(B=1, H=4, N=256, D=64, dtype="fp16", H_kv=None, seed=0):
    w = fa_inputs.Workload("bind", B, H, N, D, True, dtype)
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=seed))
    if H_kv is not None:
        k, v = k[:, :H_kv].contiguous(), v[:, :H_kv].contiguous()
    return q, k, v


def test_forward_outputs_checked():
    q, k, v = _qkv()
    B, H, N, D = q.shape
    with pytest.raises(ValueError, match="out"):
        fa.attention(q, k, v, out=torch.empty((B, H, N - 1, D), dtype=q.dtype, device="cuda"))
    with pytest.raises(ValueError, match="out"):
        fa.attention(q, k, v, out=torch.empty((B, H, N, D), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="out"):
        fa.attention(q, k, v, out=torch.empty((B, H, D, N), dtype=q.dtype, device="cuda").transpose(2, 3))
    with pytest.raises(ValueError, match="lse"):
        fa.attention(q, k, v, lse=torch.empty((B, H, N), dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError, match="workspace"):
        fa.attention(q, k, v, num_splits=2, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    # correct caller-provided outputs are written in place
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    o2, l2 = fa.attention(q, k, v, causal=True, out=out, lse=lse)
    ref_o, ref_l = fa.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert o2.data_ptr() == out.data_ptr() and torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_backward_outputs_checked():
    q, k, v = _qkv(H=8, H_kv=2)
    o, lse = fa.attention(q, k, v, causal=True)
    do = torch.randn_like(q)
    # grouped heads: dK, dV have the K/V shape, not Q's
    with pytest.raises(ValueError, match="dk"):
        fa.attention_backward(q, k, v, o, lse, do, causal=True, dk=torch.empty_like(q))
    with pytest.raises(ValueError, match="dq"):
        fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=torch.empty_like(k))
    with pytest.raises(ValueError, match="workspace"):
        fa.attention_backward(q, k, v, o, lse, do, causal=True, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    rq, rk, rv = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dk, rk) and torch.equal(dv, rv)


def test_kv_and_fp8_outputs_checked():
    q, k, v = _qkv(H=8, H_kv=2, N=512)
    qd = q[:, :, -1:].contiguous()
    with pytest.raises(ValueError, match="lse"):
        fa.attention_kv(qd, k, v, causal=True, lse=torch.empty((1, 8, 2), device="cuda"))
    with pytest.raises(ValueError, match="out"):
        fa.attention_kv(qd, k, v, causal=True, out=torch.empty_like(q))
    w = fa_inputs.Workload("bind8", 1, 2, 256, 128, True, "bf16")
    (q8, k8, v8), scs = fa_inputs.make_qkv_fp8(w, seed=1)
    q8, k8, vt = q8.cuda(), k8.cuda(), v8.transpose(2, 3).contiguous().cuda()
    scs = [t.cuda() for t in scs]
    with pytest.raises(ValueError, match="out"):
        fa.attention_fp8(q8, k8, vt, *scs, causal=True, out=torch.empty((1, 2, 256, 128), dtype=torch.float16,
                                                                         device="cuda"))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK


def test_host_outputs_checked():
    w = fa_inputs.Workload("bindh", 1, 2, 256, 64, False, "fp16")
    q, k, v = (t.pin_memory() for t in fa_inputs.make_qkv(w, seed=2))
    with pytest.raises(ValueError, match="out"):
        fa.attention_host(q, k, v, out=torch.empty(q.shape, dtype=q.dtype))            # pageable
    with pytest.raises(ValueError, match="lse"):
        fa.attention_host(q, k, v, lse=torch.empty((1, 2, 255)).pin_memory())
    with pytest.raises(ValueError, match="workspace"):
        fa.attention_host(q, k, v, workspace=torch.empty(1 << 20, dtype=torch.uint8).pin_memory())
    o, lse = fa.attention_host(q, k, v)
    od, ld = fa.attention(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
