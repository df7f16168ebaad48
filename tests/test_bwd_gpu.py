"""Parity of the CUDA backward pass (fa_bwd, through the C ABI) with the FP64
backward oracle.

Inputs are the forward's own 16-bit Q, K, V, its O and LSE from the CUDA
forward pass, and a 16-bit upstream gradient dO; the oracle differentiates
the exact attention of the same 16-bit Q, K, V with the same dO.

Tolerances.  Each gradient is compared element by element against
    c_t * max(1, max |G_ref|)
with c_fp16 = 2^-9 and c_bf16 = 2^-6: four half-ulps of the tensor's largest
element in the output type.  The error budget is the rounding of the output
itself plus the 16-bit rounding of P and dS where they enter the gradient
GEMMs (each term rounded once, accumulated in fp32).  The pages' own gradient
check (fp16, B1 H4 N1024 D64, no mask, loss = sum of O) is also run with the
pages' absolute thresholds: dQ, dK < 1e-3 and dV < 5e-3 (the FlashAttention-on-
MI50 engineering page, kwkr.cn, section 5.1, gradient consistency).
"""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

C_T = {"fp16": 2.0 ** -9, "bf16": 2.0 ** -6}


def _inputs(w, seed, ones=False):
    q, k, v = fa_inputs.make_qkv(w, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    do = (torch.ones(q.shape) if ones else torch.randn(q.shape, generator=g)).to(q.dtype)
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal, scale):
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    return dq, dk, dv


def _check(name, got, ref, dtype, what):
    x = got.float().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(x)), "%s %s: non-finite" % (what, name)
    tol = C_T[dtype] * max(1.0, float(np.abs(ref).max()))
    err = float(np.abs(x - ref).max())
    assert err <= tol, "%s %s: max err %.3e > tol %.3e" % (what, name, err, tol)
    return err


def _oracle(w, q, k, v, do):
    e = fa_inputs.enc(w)
    return fa_ref.backward(*(fa_inputs.bits(t) for t in (q, k, v, do)), w.scale, w.causal, enc=e)


def test_pages_gradient_check_case():
    """fp16 B1 H4 N1024 D64, no mask, dO = 1 (loss = O.sum())."""
    w = fa_inputs.Workload("gradcheck", 1, 4, 1024, 64, False, "fp16")
    q, k, v, do = _inputs(w, seed=0, ones=True)
    dq, dk, dv = _gpu_grads(q, k, v, do, w.causal, w.scale)
    rq, rk, rv, _ = _oracle(w, q, k, v, do)
    for name, got, ref, thr in (("dQ", dq, rq, 1e-3), ("dK", dk, rk, 1e-3), ("dV", dv, rv, 5e-3)):
        err = float(np.abs(got.float().cpu().numpy() - ref).max())
        assert err < thr, "%s max diff %.3e >= %.0e" % (name, err, thr)


SMALL_N = [1, 2, 17, 127, 128, 129, 255, 257, 300, 1000]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_shapes_fp16(N, D, causal):
    w = fa_inputs.Workload("bwd", 1, 2, N, D, causal, "fp16")
    q, k, v, do = _inputs(w, seed=N * 3 + D)
    got = _gpu_grads(q, k, v, do, causal, w.scale)
    ref = _oracle(w, q, k, v, do)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        _check(name, g, r, "fp16", "N=%d D=%d causal=%d" % (N, D, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [17, 129, 300])
def test_small_shapes_bf16(N, D, causal):
    w = fa_inputs.Workload("bwd", 1, 2, N, D, causal, "bf16")
    q, k, v, do = _inputs(w, seed=N * 5 + D)
    got = _gpu_grads(q, k, v, do, causal, w.scale)
    ref = _oracle(w, q, k, v, do)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        _check(name, g, r, "bf16", "N=%d D=%d causal=%d" % (N, D, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_batch_and_head_indexing(causal, dtype):
    w = fa_inputs.Workload("bwd_bh", 2, 3, 333, 128, causal, dtype)
    q, k, v, do = _inputs(w, seed=21)
    got = _gpu_grads(q, k, v, do, causal, w.scale)
    ref = _oracle(w, q, k, v, do)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        _check(name, g, r, dtype, "B2 H3 N333")


@pytest.mark.parametrize("name", ["causal_fp16_b1h32n4096d128", "causal_fp16_b1h32n8192d128",
                                  "noncausal_fp16_b1h32n4096d64", "peaky_causal_bf16_b2h16n16384d128"])
def test_full_size_sampled(name):
    """Full-size workloads in the bench's launch configuration: sampled dQ
    rows and sampled dK / dV keys of two heads against the oracle, plus the
    identities sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i on every head."""
    w = fa_inputs.WORKLOADS[name]
    q, k, v, do = _inputs(w, seed=0)
    dq, dk, dv = _gpu_grads(q, k, v, do, w.causal, w.scale)
    BH, N, D = w.B * w.H, w.N, w.D
    rng = np.random.default_rng(1)
    rows = np.concatenate([[0, 1, 127, 128, N // 2, N - 1], rng.integers(0, N, 58)])
    bh_q = rng.integers(0, BH, rows.size)
    heads = np.array([0, BH - 1])
    keys = np.concatenate([[0, 1, 127, 128, N // 2, N - 1], rng.integers(0, N, 26)])
    bh_k = np.repeat(heads, keys.size)
    keys = np.tile(keys, heads.size)
    e = fa_inputs.enc(w)
    rq, rk, rv = fa_ref.backward_sample(*(fa_inputs.bits(t) for t in (q, k, v, do)), w.scale, w.causal,
                                        bh_q, rows, bh_k, keys, enc=e)
    flat = lambda t: t.reshape(BH, N, D)
    dtype = w.dtype
    # each sampled gradient row against the same tolerance rule as the small shapes
    _check("dQ", flat(dq)[torch.from_numpy(bh_q).cuda(), torch.from_numpy(rows).cuda()], rq, dtype, name)
    _check("dK", flat(dk)[torch.from_numpy(bh_k).cuda(), torch.from_numpy(keys).cuda()], rk, dtype, name)
    _check("dV", flat(dv)[torch.from_numpy(bh_k).cuda(), torch.from_numpy(keys).cuda()], rv, dtype, name)
    # identities of the exact gradient, on every head (sums in fp64 of the 16-bit results)
    dkd = flat(dk).double()
    dvd = flat(dv).double()
    dod = flat(do.cuda()).double()
    assert torch.isfinite(dkd).all() and torch.isfinite(dvd).all() and torch.isfinite(flat(dq).float()).all()
    sk = dkd.sum(1).abs().max().item() / dkd.abs().sum(1).max().item()
    assert sk < 1e-2, "sum_j dK_j / sum_j |dK_j| = %.3e" % sk
    sv = (dvd.sum(1) - dod.sum(1)).abs().max().item() / dod.abs().sum(1).max().item()
    assert sv < 1e-2, "sum_j dV_j vs sum_i dO_i: %.3e" % sv


@pytest.mark.parametrize("D", [128, 64])
def test_dk_dv_deterministic_dq_close(D):
    """dK and dV are summed in TMEM in a fixed order (D = 128 in one compute pass,
    D = 64 with P and dS in two), so two runs give the same bits."""
    w = fa_inputs.Workload("det", 1, 32, 1024, D, True, "fp16")
    q, k, v, do = _inputs(w, seed=4)
    a = _gpu_grads(q, k, v, do, True, w.scale)
    b = _gpu_grads(q, k, v, do, True, w.scale)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ is summed with fp32 atomics: the order may change its last bits only
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2.0 ** -9 * max(1.0, a[0].float().abs().max().item())


def test_bad_workspace_is_rejected_before_launch():
    w = fa_inputs.Workload("ws", 1, 2, 256, 64, True, "fp16")
    q, k, v, do = (t.cuda() for t in _inputs(w, seed=2))
    o, lse = fa.attention(q, k, v, causal=True)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError):
        fa.attention_backward(q, k, v, o, lse, do, causal=True, workspace=small)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK


@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 3), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("N", [129, 300])
def test_grouped_kv_heads(N, D, dtype, causal, H, H_kv):
    """fa_bwd_gqa: the oracle's backward on K/V repeated over each group, with dK
    and dV of a K/V head the FP64 sum over the query heads that read it."""
    G = H // H_kv
    td = torch.float16 if dtype == "fp16" else torch.bfloat16
    gen = torch.Generator().manual_seed(N + 10 * H + H_kv)
    q = torch.randn(1, H, N, D, generator=gen).to(td)
    k = torch.randn(1, H_kv, N, D, generator=gen).to(td)
    v = torch.randn(1, H_kv, N, D, generator=gen).to(td)
    do = torch.randn(1, H, N, D, generator=gen).to(td)
    scale = D ** -0.5
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    assert dk.shape == k.shape and dv.shape == v.shape
    e = "f16" if dtype == "fp16" else "bf16"
    kr, vr = (t.repeat_interleave(G, dim=1) for t in (k, v))
    rq, rk, rv, _ = fa_ref.backward(*(fa_inputs.bits(t) for t in (q, kr, vr, do)), scale, causal, enc=e)
    rk = rk.reshape(1, H_kv, G, N, D).sum(axis=2)
    rv = rv.reshape(1, H_kv, G, N, D).sum(axis=2)
    what = "H%d/%d N=%d D=%d causal=%d" % (H, H_kv, N, D, causal)
    for name, g_, r_ in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _check(name, g_, r_, dtype, what)


def test_grouped_kv_heads_full_size_sampled():
    """B1 H32 H_kv 8 N4096 D128 causal fp16 (four query heads per K/V head, 32
    Q tiles each): sampled dQ rows, and sampled dK / dV keys whose reference is
    the FP64 sum over the group of the oracle's per-head gradients on repeated
    K/V."""
    B, H, H_kv, N, D, G = 1, 32, 8, 4096, 128, 4
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, N, D, generator=gen).half()
    k = torch.randn(B, H_kv, N, D, generator=gen).half()
    v = torch.randn(B, H_kv, N, D, generator=gen).half()
    do = torch.randn(B, H, N, D, generator=gen).half()
    scale = D ** -0.5
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, causal=True, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 28)])
    bh_q = rng.integers(0, B * H, rows.size)
    kv_heads = np.array([0, 3, B * H_kv - 1])
    keys = np.concatenate([[0, 1, 128, N - 1], rng.integers(0, N, 12)])
    kvh = np.repeat(kv_heads, keys.size)
    keys = np.tile(keys, kv_heads.size)
    # each K/V head's gradient is the sum over its G query heads on repeated K/V
    bh_k = (kvh[:, None] * G + np.arange(G)[None, :]).reshape(-1)
    keys_rep = np.repeat(keys, G)
    kr, vr = (t.repeat_interleave(G, dim=1) for t in (k, v))
    rq, rk, rv = fa_ref.backward_sample(*(fa_inputs.bits(t) for t in (q, kr, vr, do)), scale, True,
                                        bh_q, rows, bh_k, keys_rep, enc="f16")
    rk = rk.reshape(-1, G, D).sum(axis=1)
    rv = rv.reshape(-1, G, D).sum(axis=1)
    sel = lambda t, a, b: t.reshape(-1, N, D)[torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()]
    _check("dQ", sel(dq, bh_q, rows), rq, "fp16", "GQA full size")
    _check("dK", sel(dk, kvh, keys), rk, "fp16", "GQA full size")
    _check("dV", sel(dv, kvh, keys), rv, "fp16", "GQA full size")
