"""Parity of fa_fwd_kv (queries against a K/V sequence: decode, prefill chunks)
with the FP64 oracle's naive_kv form.  Tolerances as for the square forward
pass: max|dO| <= 2e-3 (fp16) / 1e-2 (bf16), max|dLSE| <= 1e-3."""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}


def _inputs(B, H, H_kv, Nq, Nk, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    td = torch.float16 if dtype == "fp16" else torch.bfloat16
    q = torch.randn(B, H, Nq, D, generator=g).to(td)
    k = torch.randn(B, H_kv, Nk, D, generator=g).to(td)
    v = torch.randn(B, H_kv, Nk, D, generator=g).to(td)
    return q, k, v


def _check(o, lse, q, k, v, causal, scale, dtype, what):
    e = "f16" if dtype == "fp16" else "bf16"
    o_ref, l_ref = fa_ref.naive_kv(*(fa_inputs.bits(t) for t in (q, k, v)), scale, causal, enc=e)
    of = o.float().cpu().numpy()
    assert np.all(np.isfinite(of)) and torch.isfinite(lse).all(), what
    eo = float(np.abs(of - o_ref).max())
    el = float(np.abs(lse.cpu().numpy() - l_ref).max())
    assert eo <= TOL_O[dtype] and el <= 1e-3, "%s: max|dO| %.3e max|dLSE| %.3e" % (what, eo, el)


DECODE = [  # B, H, H_kv, Nq, Nk, D
    (2, 8, 2, 1, 1, 128), (2, 8, 2, 1, 100, 128), (1, 32, 8, 1, 4096, 128), (1, 8, 1, 1, 2048, 64),
    (2, 16, 16, 1, 1000, 128), (1, 8, 2, 4, 777, 128), (3, 6, 3, 16, 5000, 64),
]


@pytest.mark.parametrize("splits", [0, 4])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", DECODE)
def test_decode_shapes(shape, causal, splits):
    B, H, H_kv, Nq, Nk, D = shape
    dtype = "bf16" if (Nk % 2) else "fp16"
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, D, dtype, seed=Nk + Nq)
    scale = D ** -0.5
    o, lse = fa.attention_kv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    _check(o, lse, q, k, v, causal, scale, dtype, "%s causal=%d splits=%d" % (shape, causal, splits))


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("shape", [(1, 4, 4, 200, 1000, 128), (1, 4, 2, 300, 1000, 64), (2, 2, 1, 129, 130, 128)])
def test_prefill_chunk_against_cache(shape, splits):
    B, H, H_kv, Nq, Nk, D = shape
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, D, "fp16", seed=Nq)
    o, lse = fa.attention_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=D ** -0.5, num_splits=splits)
    torch.cuda.synchronize()
    _check(o, lse, q, k, v, True, D ** -0.5, "fp16", "%s splits=%d" % (shape, splits))


@pytest.mark.parametrize("splits", [1, 2, 3, 5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 16, 4, 1, 5000, 128), (2, 4, 4, 128, 3000, 64), (1, 8, 8, 100, 2500, 128)])
def test_split_chunks_of_short_query_planes(shape, causal, splits):
    """Planes of at most 128 query rows (one Q tile) split into 1-5 chunks of
    K/V tiles, including chunks of odd length and the diagonal tiles of the
    end-aligned causal mask."""
    B, H, H_kv, Nq, Nk, D = shape
    dtype = "bf16" if Nq == 1 else "fp16"
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, D, dtype, seed=Nk + splits)
    o, lse = fa.attention_kv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=D ** -0.5, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    _check(o, lse, q, k, v, causal, D ** -0.5, dtype, "%s causal=%d splits=%d" % (shape, causal, splits))


def test_splits_hint_and_auto_mode():
    """The hint splits decode shapes whose unsplit grid leaves SMs idle and leaves
    large problems unsplit; num_splits="auto" gives the oracle's result."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.fa_fwd_kv_splits_hint(8, 32, 8, 1, 32768, 128, 1) == (sms // 64 if sms // 64 >= 2 else 0)
    assert fa.fa_fwd_kv_splits_hint(1, 32, 8, 1, 131072, 128, 1) == min(64, sms // 8)
    assert fa.fa_fwd_kv_splits_hint(1, 32, 32, 4096, 4096, 128, 1) == 0      # 512 work tiles
    assert fa.fa_fwd_kv_splits_hint(1, 1, 1, 32768, 32768, 128, 1) >= 2      # one long causal head
    q, k, v = _inputs(2, 16, 4, 1, 9000, 128, "bf16", seed=77)
    o, lse = fa.attention_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits="auto")
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    _check(o, lse, q, k, v, True, 128 ** -0.5, "bf16", "auto splits")


def test_long_decode_64_splits():
    q, k, v = _inputs(4, 32, 8, 1, 32768, 128, "bf16", seed=3)
    o, lse = fa.attention_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=64)
    torch.cuda.synchronize()
    _check(o, lse, q, k, v, True, 128 ** -0.5, "bf16", "B4 H32/8 Nk32768 splits=64")


@pytest.mark.parametrize("causal", [False, True])
def test_square_case_equals_fa_fwd_bitwise(causal):
    w = fa_inputs.Workload("sq", 1, 4, 700, 128, causal, "fp16")
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=5))
    o1, l1 = fa.attention(q, k, v, causal=causal)
    o2, l2 = fa.attention_kv(q, k, v, causal=causal)
    kg, vg = k[:, :2].contiguous(), v[:, :2].contiguous()
    o3, l3 = fa.attention(q, kg, vg, causal=causal)
    o4, l4 = fa.attention_kv(q, kg, vg, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o3, o4) and torch.equal(l3, l4)


def test_causal_with_more_queries_than_keys_is_rejected():
    q, k, v = (t.cuda() for t in _inputs(1, 2, 2, 10, 5, 64, "fp16", 0))
    with pytest.raises(fa.FaError):
        fa.attention_kv(q, k, v, causal=True)
