"""Seeded random shapes through the backward pass (fa_bwd / fa_bwd_gqa), every
gradient element against the FP64 oracle's backward.

24 shapes are drawn from a fixed generator: batch 1-2, query heads 1-8 with
K/V heads a divisor of them, sequence lengths 1-900, D 64 or 128, causal or
not, fp16 or bf16.  dO ~ N(0, 1).  With grouped K/V heads the oracle runs on
K/V repeated over each group and dK, dV of a K/V head are the FP64 sums over
its group.  Tolerance: every element within c_t * max(1, max |G_ref|),
c_fp16 = 2^-9, c_bf16 = 2^-6 (the backward tests' bound).
"""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

C_T = {"fp16": 2.0 ** -9, "bf16": 2.0 ** -6}


def _draws(n=24, seed=4048):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 9))
        divisors = [d for d in range(1, H + 1) if H % d == 0]
        H_kv = int(rng.choice(divisors))
        N = int(rng.choice([int(rng.integers(1, 130)), int(rng.integers(130, 900))]))
        D = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        dtype = "bf16" if rng.integers(0, 2) else "fp16"
        out.append((i, B, H, H_kv, N, D, causal, dtype))
    return out


@pytest.mark.parametrize("i,B,H,H_kv,N,D,causal,dtype", _draws())
def test_random_shape_backward_against_oracle(i, B, H, H_kv, N, D, causal, dtype):
    w = fa_inputs.Workload("rndb%d" % i, B, H, N, D, causal, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=300 + i)
    k, v = k[:, :H_kv].contiguous(), v[:, :H_kv].contiguous()
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(400 + i)).to(q.dtype)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    g = H // H_kv
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    rq, rk, rv, _ = fa_ref.backward(*(fa_inputs.bits(t) for t in (q, kr, vr, do)), w.scale, causal,
                                    enc=fa_inputs.enc(w))
    rk = rk.reshape(B, H_kv, g, N, D).sum(axis=2)
    rv = rv.reshape(B, H_kv, g, N, D).sum(axis=2)
    what = "B%d H%d/%d N%d D%d causal=%d %s" % (B, H, H_kv, N, D, causal, dtype)
    for name, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        x = got.float().cpu().numpy().reshape(ref.shape)
        assert np.all(np.isfinite(x)), "%s %s: non-finite" % (what, name)
        tol = C_T[dtype] * max(1.0, float(np.abs(ref).max()))
        err = float(np.abs(x - ref).max())
        assert err <= tol, "%s %s: max err %.3e > tol %.3e" % (what, name, err, tol)
