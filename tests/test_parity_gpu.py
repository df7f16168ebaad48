"""Parity of the CUDA path (through the C ABI) with the FP64 oracle.

Every output element is compared with the oracle: small shapes, shapes with
more work tiles than two rounds of the persistent grid, and every full-size
workload, run in the launch configuration the bench uses (the oracle runs on
all host cores; the full-size workloads take it a few minutes together).  For
those, the errors are also recorded (max-abs, RMS and relative L2 of O,
max-abs of the LSE, and the output type's rounding floor) in the JSON-lines
file named by the FA_ACCURACY_OUT environment variable, when it is set.
Tolerances (against the FP64 oracle on the
same 16-bit-rounded inputs): max |dO| <= 2e-3 for fp16 outputs, <= 1e-2 for
bf16 outputs, max |dLSE| <= 1e-3.  For the peaky bf16 workload (scores with
a standard deviation of 9, not N(0,1) inputs) the bf16 rounding of O alone
can exceed 1e-2 where |O| >= 4, so each element there may also use half a
bf16 ulp of the exact value on top of 1e-2.
"""
import json
import os
import time

import numpy as np
import pytest
import torch

import bench
import exact_attention_22_gb300 as fa
import fa_inputs
from oracle import fa_ref

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3


def _run(q, k, v, causal, scale, stream=None):
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, stream=stream)
    torch.cuda.synchronize()
    return o, lse


def _bf16_half_ulp(x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - 7)


def _check(o, lse, o_ref, lse_ref, dtype, peaky=False, what=""):
    o = o.float().cpu().numpy().reshape(o_ref.shape)
    lse = lse.cpu().numpy().reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    err = np.abs(o - o_ref)
    tol = TOL_O[dtype] + (_bf16_half_ulp(o_ref) if peaky else 0.0)
    bad = err > tol
    assert not bad.any(), "%s: %d elements over tolerance, max|dO|=%.3e" % (what, bad.sum(), err.max())
    el = np.abs(lse - lse_ref).max()
    assert el <= TOL_LSE, "%s: max|dLSE|=%.3e" % (what, el)
    return float(err.max()), float(el)


def _oracle_full(q, k, v, causal, scale):
    e = fa_inputs.enc(q.dtype)
    return fa_ref.naive(fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v), scale, causal, enc=e)


SMALL_N = [1, 2, 3, 17, 127, 128, 129, 255, 256, 257, 300, 511, 1000]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_shapes_elementwise(N, D, causal, dtype):
    w = fa_inputs.Workload("small", 1, 2, N, D, causal, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=N * 7 + D)
    o, lse = _run(q, k, v, causal, w.scale)
    o_ref, lse_ref = _oracle_full(q, k, v, causal, w.scale)
    _check(o, lse, o_ref, lse_ref, dtype, what="N=%d D=%d causal=%d %s" % (N, D, causal, dtype))


@pytest.mark.parametrize("causal", [False, True])
def test_batch_and_head_indexing(causal):
    w = fa_inputs.Workload("bh", 2, 3, 333, 128, causal, "bf16")
    q, k, v = fa_inputs.make_qkv(w, seed=5)
    o, lse = _run(q, k, v, causal, w.scale)
    o_ref, lse_ref = _oracle_full(q, k, v, causal, w.scale)
    _check(o, lse, o_ref, lse_ref, "bf16", what="B2 H3 N333")


def test_tiny_workload_elementwise():
    w = fa_inputs.WORKLOADS["tiny_fp16_b1h2n256d64"]
    q, k, v = fa_inputs.make_qkv(w, seed=0)
    o, lse = _run(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = _oracle_full(q, k, v, w.causal, w.scale)
    _check(o, lse, o_ref, lse_ref, w.dtype, what=w.name)


# With no more 256-row work tiles than SMs, fa_fwd deals 128-row Q tiles whose
# K/V tiles are shared out between the CTA's two streams (ceil(J/2) and
# floor(J/2) of J) and merges the two partial (m, l, O) on chip.  These shapes
# cover: a Q tile with one K/V tile (stream 1 has none), odd and even J, a ragged
# last tile, grouped K/V heads, and the edge between the two forms on a 152-SM
# GB300 (B1 H38 N1024: 152 tiles, key split; H39: 156 tiles, 256-row tiles).
@pytest.mark.parametrize("B,H,H_kv,N,D,causal,dtype", [
    (1, 4, 4, 129, 128, True, "fp16"),
    (1, 3, 3, 640, 64, True, "bf16"),
    (2, 5, 5, 1000, 128, False, "fp16"),
    (1, 8, 2, 777, 64, True, "fp16"),
    (1, 38, 38, 1024, 128, True, "fp16"),
    (1, 39, 39, 1024, 128, True, "fp16"),
])
def test_key_split_and_its_edge_elementwise(B, H, H_kv, N, D, causal, dtype):
    w = fa_inputs.Workload("ks", B, H, N, D, causal, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=11)
    k, v = k[:, :H_kv].contiguous(), v[:, :H_kv].contiguous()
    o, lse = _run(q, k, v, causal, w.scale)
    g = H // H_kv
    o_ref, lse_ref = _oracle_full(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1), causal, w.scale)
    _check(o, lse, o_ref, lse_ref, dtype, what="B%d H%d/%d N%d D%d" % (B, H, H_kv, N, D))


@pytest.mark.parametrize("B,H,N,D,causal,dtype", [
    (2, 32, 2048, 128, True, "fp16"),    # 512 work tiles: 3.4 rounds of the persistent grid
    (4, 16, 1024, 64, False, "bf16"),    # 256 work tiles, every CTA past its first round
    (3, 40, 1280, 128, False, "fp16"),   # 600 work tiles, N a multiple of 256
])
def test_multi_round_persistent_elementwise(B, H, N, D, causal, dtype):
    """More work tiles than two rounds of one CTA per SM: the snake order and
    the early first S of a CTA's next work tile are compared element by
    element."""
    w = fa_inputs.Workload("rounds", B, H, N, D, causal, dtype)
    q, k, v = fa_inputs.make_qkv(w, seed=B * 100 + H)
    o, lse = _run(q, k, v, causal, w.scale)
    o_ref, lse_ref = _oracle_full(q, k, v, causal, w.scale)
    _check(o, lse, o_ref, lse_ref, dtype, what="B%d H%d N%d D%d" % (B, H, N, D))


def _sample_rows(w, n_random=192, seed=0):
    """Rows of a large problem for the oracle to evaluate one by one (used by
    the split-K tests): the tile edges and the ends, plus random rows."""
    rng = np.random.default_rng(seed)
    N, BH = w.N, w.B * w.H
    special = [0, 1, 2, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128, N - 2, N - 1]
    special = sorted({r for r in special if 0 <= r < N})
    rows, bhs = [], []
    for i, r in enumerate(special):
        rows.append(r)
        bhs.append(i % BH)
    rows += list(rng.integers(0, N, n_random))
    bhs += list(rng.integers(0, BH, n_random))
    return np.array(bhs, np.int64), np.array(rows, np.int64)


def _record(entry):
    path = os.environ.get("FA_ACCURACY_OUT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(entry) + "\n")


@pytest.mark.parametrize("name", sorted(n for n in fa_inputs.WORKLOADS if not n.startswith("tiny")))
def test_full_size_workloads_every_row(name):
    w = fa_inputs.WORKLOADS[name]
    q, k, v = fa_inputs.make_qkv(w, seed=0)
    o, lse = _run(q, k, v, w.causal, w.scale)
    assert fa.fa_get_device_status(0) == fa.FA_OK
    t0 = time.perf_counter()
    o_ref, lse_ref = _oracle_full(q, k, v, w.causal, w.scale)
    secs = time.perf_counter() - t0
    peaky = w.qk_std != 1.0
    stats = bench.accuracy_stats(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, w.dtype)
    stats.update(workload=name, seed=0, oracle_seconds=secs, oracle_threads=fa_ref.max_threads(),
                 literal_gate_o=TOL_O[w.dtype],
                 over_literal_gate=int((np.abs(o.float().cpu().numpy().reshape(o_ref.shape) - o_ref)
                                        > TOL_O[w.dtype]).sum()))
    _record(stats)
    _check(o, lse, o_ref, lse_ref, w.dtype, peaky=peaky, what=name)
    if w.causal:
        assert torch.equal(o[:, :, 0, :].cpu(), v[:, :, 0, :])   # row 0 sees only key 0


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_values(causal, dtype):
    w = fa_inputs.Workload("uni", 1, 2, 700, 128, causal, dtype)
    _, k, v = fa_inputs.make_qkv(w, seed=3)
    q = torch.zeros_like(k)
    o, lse = _run(q, k, v, causal, w.scale)
    vd = v.double()
    if causal:
        want = vd.cumsum(2) / torch.arange(1, w.N + 1, dtype=torch.float64).view(1, 1, -1, 1)
        want_lse = torch.log(torch.arange(1, w.N + 1, dtype=torch.float64)).expand(1, 2, -1)
    else:
        want = vd.mean(2, keepdim=True).expand_as(vd)
        want_lse = torch.full((1, 2, w.N), float(np.log(w.N)), dtype=torch.float64)
    _check(o, lse, want.numpy(), want_lse.numpy(), dtype, what="uniform")


@pytest.mark.parametrize("causal", [False, True])
def test_extreme_inputs_stay_finite(causal):
    """fp16 max and mixed +-1e4 entries: the max subtraction keeps O finite."""
    w = fa_inputs.Workload("ext", 1, 1, 300, 64, causal, "fp16")
    g = torch.Generator().manual_seed(11)
    choice = torch.tensor([-1e4, 1e4, 65504.0, 0.5], dtype=torch.float16)
    q = choice[torch.randint(0, 4, (1, 1, 300, 64), generator=g)]
    k = choice[torch.randint(0, 4, (1, 1, 300, 64), generator=g)]
    v = torch.randn(1, 1, 300, 64, generator=g).half()
    o, lse = _run(q, k, v, causal, 1.0 / 8)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    vmax, vmin = v.float().amax(2, keepdim=True).cuda(), v.float().amin(2, keepdim=True).cuda()
    assert (o.float() <= vmax + 1e-3).all() and (o.float() >= vmin - 1e-3).all()


def test_deterministic_and_stream_aware():
    w = fa_inputs.WORKLOADS["causal_fp16_b1h32n1024d128"]
    q, k, v = (t.cuda() for t in fa_inputs.make_qkv(w, seed=1))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = fa.attention(q, k, v, causal=True, stream=s)
        o2, l2 = fa.attention(q, k, v, causal=True, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert fa.fa_get_device_status(s.cuda_stream) == fa.FA_OK


def test_bad_arguments_leave_outputs_untouched():
    q = torch.randn(1, 1, 64, 96, device="cuda", dtype=torch.float16)
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 64), 7.0, device="cuda")
    st = fa.fa_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 64, 96, 0.1, 0,
                   fa.FA_FP16, 0)
    assert st == 2
    torch.cuda.synchronize()
    assert (o == 7).all() and (lse == 7).all()
    assert fa.fa_get_device_status(0) == fa.FA_OK


def test_bounded_wait_gives_up_and_context_survives():
    """A wait that nothing completes gives up after its limit and is reported
    as FA_ERR_TIMEOUT; the next forward pass on the same context is correct."""
    import time
    s = torch.cuda.Stream()
    t0 = time.time()
    assert fa.fa_selftest_wait_timeout(s.cuda_stream) == fa.FA_OK
    assert fa.fa_get_device_status(s.cuda_stream) == 5          # FA_ERR_TIMEOUT
    assert 0.5 < time.time() - t0 < 30
    assert fa.fa_get_device_status(s.cuda_stream) == fa.FA_OK   # reading clears it
    w = fa_inputs.Workload("after", 1, 2, 300, 64, True, "fp16")
    q, k, v = fa_inputs.make_qkv(w, seed=9)
    o, lse = _run(q, k, v, True, w.scale)
    o_ref, lse_ref = _oracle_full(q, k, v, True, w.scale)
    _check(o, lse, o_ref, lse_ref, "fp16", what="after self-test")
