"""Pins of the FP64 backward oracle (oracle/fa_ref.c, fa_ref_backward*).

The oracle follows the gradient formulas of "Why FlashAttention does not need
to store the attention matrix" (section 3.3) and "CUDA FlashAttention: from
online softmax to the long-sequence IO limit" (section 4.3.1).  These tests
tie it to things other than those formulas:

* central finite differences of the pinned forward oracle (the gradient is
  the derivative of the forward definition, whatever formula computes it);
* float64 autograd of a plain softmax(Q K^T * scale + mask) V written in
  torch ops, an independent derivation of the same gradient;
* identities the exact gradient satisfies: sum_j dK_j = 0 (softmax is
  invariant to a shift of a row's scores), sum_j dV_j = sum_i dO_i (each P row
  sums to 1), Delta_i = dO_i . O_i;
* closed forms when every score of a row is equal (Q = 0) and for causal
  row 0, which sees one key only.
"""
import numpy as np
import pytest
import torch

import fa_inputs
from oracle import fa_ref


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return [scale * rng.normal(size=shape) for _ in range(4)]


def _loss(q, k, v, g, scale, causal):
    o, _ = fa_ref.naive(q, k, v, scale, causal)
    return float(np.sum(o * g))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,D", [(1, 3), (2, 4), (5, 3), (9, 4)])
def test_finite_differences(N, D, causal):
    q, k, v, g = _rand((1, 1, N, D), seed=N * 10 + D)
    scale = 0.7
    dq, dk, dv, _ = fa_ref.backward(q, k, v, g, scale, causal)
    h = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, g, scale, causal)
            x[idx] = old - h
            lm = _loss(q, k, v, g, scale, causal)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max()
        assert err <= 1e-8 * (1 + np.abs(grad).max()), "d%s: max |fd - oracle| = %.3e" % (name, err)


def _torch_grads(q, k, v, g, scale, causal):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.matmul(torch.softmax(s, dim=-1), vt)
    o.backward(torch.tensor(g, dtype=torch.float64))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_float64_autograd(causal):
    q, k, v, g = _rand((2, 2, 37, 16), seed=3)
    scale = 0.25
    dq, dk, dv, _ = fa_ref.backward(q, k, v, g, scale, causal)
    tq, tk, tv = _torch_grads(q, k, v, g, scale, causal)
    for name, a, b in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
        assert np.abs(a - b).max() <= 1e-12 * (1 + np.abs(b).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_identities(causal):
    q, k, v, g = _rand((1, 3, 200, 32), seed=7)
    scale = 32 ** -0.5
    dq, dk, dv, delta = fa_ref.backward(q, k, v, g, scale, causal)
    o, _ = fa_ref.naive(q, k, v, scale, causal)
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12 * np.abs(dk).sum()
    assert np.abs(dv.sum(axis=2) - g.sum(axis=2)).max() <= 1e-11
    assert np.abs(delta - np.sum(g * o, axis=-1)).max() <= 1e-12 * (1 + np.abs(delta).max())


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_closed_form(causal):
    _, k, v, g = _rand((1, 2, 50, 8), seed=11)
    q = np.zeros_like(k)
    scale = 0.5
    dq, dk, dv, _ = fa_ref.backward(q, k, v, g, scale, causal)
    N = q.shape[2]
    assert np.all(dk == 0.0)   # dK = scale * dS^T Q with Q = 0
    want_dq = np.zeros_like(dq)
    want_dv = np.zeros_like(dv)
    for i in range(N):
        vis = np.arange(i + 1) if causal else np.arange(N)
        n = len(vis)
        vbar = v[:, :, vis].mean(axis=2)                                   # [B,H,D]
        w = np.einsum("bhd,bhjd->bhj", g[:, :, i], v[:, :, vis] - vbar[:, :, None])
        want_dq[:, :, i] = scale / n * np.einsum("bhj,bhjd->bhd", w, k[:, :, vis])
        want_dv[:, :, vis] += g[:, :, i][:, :, None, :] / n
    assert np.abs(dq - want_dq).max() <= 1e-12
    assert np.abs(dv - want_dv).max() <= 1e-12


def test_causal_row0_has_no_query_gradient():
    q, k, v, g = _rand((1, 2, 40, 16), seed=13)
    dq, _, _, delta = fa_ref.backward(q, k, v, g, 0.3, True)
    assert np.all(dq[:, :, 0] == 0.0)
    # row 0 sees key 0 alone: P_00 = 1, so Delta_0 = dO_0 . v_0
    assert np.abs(delta[:, :, 0] - np.sum(g[:, :, 0] * v[:, :, 0], axis=-1)).max() <= 1e-13


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_16bit_inputs_decode_exactly(dtype):
    w = fa_inputs.Workload("bwd16", 1, 2, 64, 32, True, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=2)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(q.dtype)
    e = fa_inputs.enc(w)
    a = fa_ref.backward(*(fa_inputs.bits(t) for t in (q, k, v, g)), w.scale, True, enc=e)
    b = fa_ref.backward(*(t.double().numpy() for t in (q, k, v, g)), w.scale, True, enc="f64")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_entries_match_full(causal):
    q, k, v, g = _rand((2, 2, 70, 8), seed=17)
    dq, dk, dv, _ = fa_ref.backward(q, k, v, g, 0.4, causal)
    bh_q, rows = np.array([0, 3, 2, 1]), np.array([0, 69, 33, 5])
    bh_k, keys = np.array([3, 0, 1]), np.array([69, 0, 40])
    sq, sk, sv = fa_ref.backward_sample(q, k, v, g, 0.4, causal, bh_q, rows, bh_k, keys)
    flat = lambda t: t.reshape(4, 70, 8)
    assert np.array_equal(sq, flat(dq)[bh_q, rows])
    assert np.array_equal(sk, flat(dk)[bh_k, keys])
    assert np.array_equal(sv, flat(dv)[bh_k, keys])
