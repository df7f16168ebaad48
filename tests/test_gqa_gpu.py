"""Grouped K/V heads (fa_fwd_gqa): query head h reads K/V head h / (H/H_kv),
against the FP64 oracle's grouped form."""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref
from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def _qkv(B, H, H_kv, N, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.float16 if dtype == "fp16" else torch.bfloat16
    q = torch.randn(B, H, N, D, generator=g).to(dt)
    k = torch.randn(B, H_kv, N, D, generator=g).to(dt)
    v = torch.randn(B, H_kv, N, D, generator=g).to(dt)
    return q, k, v


@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 3), (4, 1), (4, 4)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("N", [129, 640])
def test_gqa_elementwise(N, D, dtype, causal, H, H_kv):
    B = 2
    q, k, v = _qkv(B, H, H_kv, N, D, dtype, seed=N + H * 7 + H_kv)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=D ** -0.5)
    torch.cuda.synchronize()
    e = fa_inputs.enc(q.dtype)
    o_ref, lse_ref = fa_ref.naive_gqa(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), D ** -0.5, causal,
                                      enc=e)
    _check(o, lse, o_ref, lse_ref, dtype, what="gqa H=%d H_kv=%d N=%d" % (H, H_kv, N))


def test_gqa_matches_fa_fwd_on_repeated_kv():
    """The grouped entry and fa_fwd on explicitly repeated K/V heads run the
    same tiles on the same data: the outputs are bit-identical."""
    B, H, H_kv, N, D = 1, 32, 4, 2048, 128
    q, k, v = (t.cuda() for t in _qkv(B, H, H_kv, N, D, "fp16", seed=1))
    o1, l1 = fa.attention(q, k, v, causal=True)
    rep = H // H_kv
    o2, l2 = fa.attention(q, k.repeat_interleave(rep, 1).contiguous(), v.repeat_interleave(rep, 1).contiguous(),
                          causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_argument_errors():
    q = torch.zeros(1, 6, 128, 64, device="cuda", dtype=torch.float16)
    k = torch.zeros(1, 4, 128, 64, device="cuda", dtype=torch.float16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 6, 128, device="cuda")
    args = (q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr())
    assert fa.fa_fwd_gqa(*args, 1, 6, 4, 128, 64, 0.125, 0, 0, 0) == 1      # 4 does not divide 6
    assert fa.fa_fwd_gqa(*args, 1, 6, 0, 128, 64, 0.125, 0, 0, 0) == 1
    assert fa.fa_fwd_gqa(*args, 1, 6, 3, 128, 96, 0.125, 0, 0, 0) == 2
    with pytest.raises(ValueError):
        fa.attention(q, k, k)
