"""Split-K forward (fa_fwd_splitkv): partials over chunks of each query
block's key/value range, merged by a second kernel, against the FP64 oracle.
The merged result is the exact attention, so the tolerances are those of
fa_fwd."""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref
from test_parity_gpu import _check, _oracle_full, _sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16"), (128, "fp16")])
@pytest.mark.parametrize("N", [1, 129, 700, 1000])
def test_splitkv_elementwise(N, D, dtype, causal, splits):
    w = fa_inputs.Workload("split", 1, 2, N, D, causal, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=N + splits)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale, num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = _oracle_full(q, k, v, causal, w.scale)
    _check(o, lse, o_ref, lse_ref, dtype, what="split N=%d D=%d causal=%d %s S=%d" % (N, D, causal, dtype, splits))


def test_splitkv_matches_unsplit_closely():
    """Same inputs through fa_fwd and fa_fwd_splitkv: both are the exact
    attention; they differ only by rounding order."""
    w = fa_inputs.WORKLOADS["causal_fp16_b1h32n1024d128"]
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=2))
    o1, l1 = fa.attention(q, k, v, causal=True)
    o2, l2 = fa.attention(q, k, v, causal=True, num_splits=4)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-3
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_splitkv_long_context_sampled_rows():
    w = fa_inputs.WORKLOADS["ragged_causal_bf16_b1h8n32749d128"]
    q, k, v = fa_inputs.make_qkv(w, seed=0)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=8)
    torch.cuda.synchronize()
    bh, rows = _sample_rows(w)
    o_ref, lse_ref = fa_ref.naive_rows(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), w.scale, True, bh,
                                       rows, enc="bf16")
    idx = (torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda())
    _check(o.reshape(8, w.N, w.D)[idx], lse.reshape(8, w.N)[idx], o_ref, lse_ref, "bf16", what="split 32749")


def test_splitkv_argument_errors():
    B, H, N, D = 1, 2, 256, 64
    assert fa.fa_splitkv_workspace_bytes(B, H, N, D, 4) == 4 * B * H * N * (4 * D + 16)
    assert fa.fa_splitkv_workspace_bytes(B, H, N, D, 0) == 0
    assert fa.fa_splitkv_workspace_bytes(B, H, N, D, 65) == 0
    q = torch.randn(B, H, N, D, device="cuda", dtype=torch.float16)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    need = fa.fa_splitkv_workspace_bytes(B, H, N, D, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, D, 0.125, 0, 0)
    assert fa.fa_fwd_splitkv(*args, 4, ws.data_ptr(), need - 16, 0) == 1      # too small
    assert fa.fa_fwd_splitkv(*args, 0, ws.data_ptr(), need, 0) == 1           # no split
    assert fa.fa_fwd_splitkv(*args, 4, 0, need, 0) == 3                       # null
    assert fa.fa_fwd_splitkv(*args, 4, ws.data_ptr() + 8, need, 0) == 3       # misaligned
    assert fa.fa_fwd_splitkv(*args, 4, o.data_ptr(), need, 0) == 1            # overlaps o
    assert fa.fa_fwd_splitkv(*args, 4, ws.data_ptr(), need, 0) == 0
    assert fa.fa_get_device_status(0) == fa.FA_OK


@pytest.mark.parametrize("splits", [4, 6, 8, 16])
def test_splitkv_causal_many_short_chunks(splits):
    """Causal with many work tiles per CTA and short chunks: chunks where one
    stream has no keys change the order in which the two streams read a K/V
    slot.  Sampled rows against the oracle, and two runs bit-identical."""
    w = fa_inputs.WORKLOADS["causal_fp16_b1h32n4096d128"]
    q, k, v = fa_inputs.make_qkv(w, seed=3)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.attention(qc, kc, vc, causal=True, num_splits=splits)
    o2, lse2 = fa.attention(qc, kc, vc, causal=True, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    bh, rows = _sample_rows(w, n_random=256, seed=splits)
    o_ref, lse_ref = fa_ref.naive_rows(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), w.scale, True, bh,
                                       rows, enc="f16")
    idx = (torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda())
    _check(o.reshape(32, w.N, w.D)[idx], lse.reshape(32, w.N)[idx], o_ref, lse_ref, "fp16", what="S=%d" % splits)


def test_splitkv_single_long_head_sampled_rows():
    """The regime split-K is for: one head, N = 32768, causal."""
    w = fa_inputs.WORKLOADS["longhead_causal_bf16_b1h1n32768d128"]
    q, k, v = fa_inputs.make_qkv(w, seed=0)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=4)
    torch.cuda.synchronize()
    bh, rows = _sample_rows(w)
    o_ref, lse_ref = fa_ref.naive_rows(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), w.scale, True, bh,
                                       rows, enc="bf16")
    idx = (torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda())
    _check(o.reshape(1, w.N, w.D)[idx], lse.reshape(1, w.N)[idx], o_ref, lse_ref, "bf16", what="split long head")
