"""Parity of the FP8 forward pass (fa_fwd_fp8, through the C ABI) with the FP64
oracle on the dequantized inputs.

Inputs are N(0,1) Q, K, V quantized per 128-row block to OCP E4M3
(fa_inputs.quantize_e4m3_blocks); the oracle decodes the same bytes and
multiplies by the same block scales, then evaluates exact attention.  The
quantization of Q, K, V is therefore not an error here; what differs is the
rounding of P to E4M3 for the FP8 product P V.

Tolerance for O, element by element.  With p~_j = p_j (1 + e_j), |e_j| <= u =
2^-4 (half an ulp of a 3-bit mantissa), O normalised by the sum of the p~ is a
convex combination with weights w~_j, and
    |O~ - O| = |sum_j (w~_j - w_j)(v_j - O)| <= 2u/(1-u) * sum_j w_j |v_j - O|,
per output element (d).  The test allows twice that (probabilities that fall
into E4M3's subnormal range have a larger relative error, and fp32 effects),
plus the bf16 rounding of the output (8 significant bits: at most 2^-8 |O|)
and 1e-4.
The LSE comes from the unrounded sums: |dLSE| <= 1e-4.
"""
import numpy as np
import pytest
import torch

import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

U = 2.0 ** -4


def _gpu(w, seed):
    (q8, k8, v8), (qs, ks, vs) = fa_inputs.make_qkv_fp8(w, seed=seed)
    v8t = v8.transpose(2, 3).contiguous()
    o, lse = fa.attention_fp8(q8.cuda(), k8.cuda(), v8t.cuda(), qs.cuda(), ks.cuda(), vs.cuda(), causal=w.causal,
                              scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == fa.FA_OK
    deq = [fa_ref.dequant_e4m3(x.numpy(), s.numpy()) for x, s in ((q8, qs), (k8, ks), (v8, vs))]
    return o, lse, deq


def _bound_rows(qd, kd, vd, scale, causal, bh, rows, o_ref):
    """2 * 2u/(1-u) * sum_j w_j |v_j - O| per (row, d), float64."""
    BH, N, D = qd.shape[0] * qd.shape[1], qd.shape[2], qd.shape[3]
    q, k, v = (x.reshape(BH, N, D) for x in (qd, kd, vd))
    out = np.empty((len(rows), D))
    for r, (h, i) in enumerate(zip(bh, rows)):
        nv = i + 1 if causal else N
        s = scale * (k[h, :nv] @ q[h, i])
        wgt = np.exp(s - s.max())
        wgt /= wgt.sum()
        out[r] = wgt @ np.abs(v[h, :nv] - o_ref[r])
    return 2.0 * 2 * U / (1 - U) * out


def _check(o, lse, o_ref, lse_ref, bound, what):
    o = o.float().cpu().numpy().reshape(o_ref.shape)
    lse = lse.cpu().numpy().reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    tol = bound + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    err = np.abs(o - o_ref)
    bad = err > tol
    assert not bad.any(), "%s: %d of %d elements over the bound, worst err/tol %.3f" % (
        what, bad.sum(), bad.size, float((err / tol).max()))
    el = float(np.abs(lse - lse_ref).max())
    assert el <= 1e-4, "%s: max|dLSE| = %.3e" % (what, el)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [16, 128, 144, 512, 1008])
def test_small_shapes(N, causal):
    w = fa_inputs.Workload("fp8", 1, 2, N, 128, causal, "bf16")
    o, lse, (qd, kd, vd) = _gpu(w, seed=N)
    o_ref, lse_ref = fa_ref.naive(qd, kd, vd, w.scale, causal)
    bh = np.repeat(np.arange(2), N)
    rows = np.tile(np.arange(N), 2)
    bound = _bound_rows(qd, kd, vd, w.scale, causal, bh, rows, o_ref.reshape(-1, 128))
    _check(o, lse, o_ref.reshape(-1, 128), lse_ref.reshape(-1), bound, "N=%d causal=%d" % (N, causal))


def test_peaky_scores_and_batches():
    w = fa_inputs.Workload("fp8_peaky", 2, 3, 1024, 128, True, "bf16", qk_std=3.0)
    o, lse, (qd, kd, vd) = _gpu(w, seed=7)
    o_ref, lse_ref = fa_ref.naive(qd, kd, vd, w.scale, True)
    rng = np.random.default_rng(0)
    bh = rng.integers(0, 6, 256)
    rows = rng.integers(0, 1024, 256)
    o_s = o.reshape(6, 1024, 128)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    l_s = lse.reshape(6, 1024)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    o_r = o_ref.reshape(6, 1024, 128)[bh, rows]
    l_r = lse_ref.reshape(6, 1024)[bh, rows]
    _check(o_s, l_s, o_r, l_r, _bound_rows(qd, kd, vd, w.scale, True, bh, rows, o_r), "peaky")


def test_full_size_sampled_rows():
    """The bench workload's shape (B1 H32 N8192 D128 causal) in FP8, sampled rows."""
    w = fa_inputs.Workload("fp8_bench", 1, 32, 8192, 128, True, "bf16")
    o, lse, (qd, kd, vd) = _gpu(w, seed=0)
    rng = np.random.default_rng(2)
    rows = np.concatenate([[0, 1, 127, 128, 4095, 8191], rng.integers(0, 8192, 90)])
    bh = rng.integers(0, 32, rows.size)
    o_r, l_r = fa_ref.naive_rows(qd, kd, vd, w.scale, True, bh, rows)
    o_s = o.reshape(32, 8192, 128)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    l_s = lse.reshape(32, 8192)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    _check(o_s, l_s, o_r, l_r, _bound_rows(qd, kd, vd, w.scale, True, bh, rows, o_r), "B1 H32 N8192")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_per_block_scales_are_applied():
    """Scaling Q's, K's or V's block scales (with the bytes unchanged) must act
    like scaling the dequantized tensor: V scale x2 doubles O, K scale x2
    doubles the scores."""
    w = fa_inputs.Workload("fp8_scales", 1, 2, 384, 128, False, "bf16")
    (q8, k8, v8), (qs, ks, vs) = fa_inputs.make_qkv_fp8(w, seed=11)
    v8t = v8.transpose(2, 3).contiguous()
    args = lambda a, b, c: fa.attention_fp8(q8.cuda(), k8.cuda(), v8t.cuda(), a.cuda(), b.cuda(), c.cuda(),
                                            causal=False, scale=w.scale)
    o1, l1 = args(qs, ks, vs)
    o2, l2 = args(qs, ks, vs * 2)
    torch.cuda.synchronize()
    assert torch.allclose(o2.float(), 2 * o1.float(), rtol=2 ** -7, atol=1e-3)
    assert torch.equal(l1, l2)
    o3, l3 = args(qs, ks * 2, vs)
    qd, kd, vd = (fa_ref.dequant_e4m3(x.numpy(), s.numpy()) for x, s in ((q8, qs), (k8, ks * 2), (v8, vs)))
    _, lse_ref = fa_ref.naive(qd, kd, vd, w.scale, False)
    assert float(np.abs(l3.cpu().numpy() - lse_ref).max()) <= 1e-4


def test_argument_errors_leave_outputs_untouched():
    q = torch.zeros(1, 1, 100, 128, dtype=torch.uint8, device="cuda")   # N = 100 is not a multiple of 16
    sc = torch.ones(1, 1, 1, device="cuda")
    o = torch.full((1, 1, 100, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 1, 100), 7.0, device="cuda")
    vt = torch.zeros(1, 1, 128, 100, dtype=torch.uint8, device="cuda")
    st = fa.fa_fwd_fp8(q.data_ptr(), q.data_ptr(), vt.data_ptr(), sc.data_ptr(), sc.data_ptr(), sc.data_ptr(),
                       o.data_ptr(), lse.data_ptr(), 1, 1, 100, 128, 0.1, 0, 0)
    assert st == 1
    st = fa.fa_fwd_fp8(q.data_ptr(), q.data_ptr(), vt.data_ptr(), sc.data_ptr(), sc.data_ptr(), sc.data_ptr(),
                       o.data_ptr(), lse.data_ptr(), 1, 1, 96, 64, 0.1, 0, 0)
    assert st == 2
    torch.cuda.synchronize()
    assert (o == 7).all() and (lse == 7).all()
