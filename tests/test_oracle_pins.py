"""Pins of the FP64 oracle to facts fixed by the pages and by mathematics.

None of these tests compares the oracle with itself: each checks a value a
page prints (fixtures under tests/golden/), a closed form, an invariant, an
exact special case, or an independent library route on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from golden_io import kv, table
from oracle import fa_ref


def _normal(seed, N, D):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(N, D)), rng.normal(size=(N, D)), rng.normal(size=(N, D))


def test_worked_row_split():
    """mpbf.cn/news/61284, section 2.2: row [1,2,3,4] merged as [1,2] | [3,4]."""
    g = kv("worked_row_split.txt")
    scores = [float(x) for x in g["scores"].split()]
    N = len(scores)
    q = np.zeros((N, 1)); q[0, 0] = 1.0
    k = np.array(scores).reshape(N, 1)
    v = np.ones((N, 1))
    _, lse, tr, _ = fa_ref.blocked(q, k, v, 1.0, Br=1, Bc=int(g["block_split"]),
                                   kv_outer=True, trace_row=0)
    assert tr.shape == (2, 4)
    # exact values of the merge
    assert tr[0, 1] == 2.0 and tr[1, 1] == 4.0
    assert abs(tr[0, 2] - (math.exp(-1) + 1)) < 1e-15
    assert abs(tr[1, 2] - ((math.exp(-1) + 1) * math.exp(-2) + math.exp(-1) + 1)) < 1e-15
    assert tr[0, 3] == 0.0 and abs(tr[1, 3] - math.exp(-2)) < 1e-16
    # the page's printed, rounded values
    dec = int(g["printed_decimals"])
    assert tr[0, 1] == float(g["block1_ref_max"]) and tr[1, 1] == float(g["block2_ref_max"])
    assert round(tr[0, 2], dec) == float(g["block1_sum"])
    assert round(tr[1, 3], dec) == float(g["block2_rescale"])
    assert round(tr[1, 2], dec) == float(g["block2_sum"])
    # the final LSE of row 0 is the max plus the log of the running sum
    assert abs(lse[0, 0, 0] - (4.0 + math.log(tr[1, 2]))) < 1e-15


def test_recurrence_trace_matches_printed():
    """'Why FlashAttention does not need to store the attention matrix', 4.1."""
    want = table("recurrence_trace_n8_d4_bc2.txt")
    Q, K, V = _normal(0, 8, 4)
    _, _, tr, _ = fa_ref.blocked(Q, K, V, 0.5, Br=8, Bc=2, kv_outer=True, trace_row=0)
    assert tr.shape == (len(want), 4)
    for got, exp in zip(tr, want):
        assert got[0] == exp[0]
        for a, b in zip(got[1:], exp[1:]):
            assert abs(a - b) <= 5.01e-5, (got, exp)


@pytest.mark.parametrize("row", table("exactness_table.txt"), ids=lambda r: "N%d_c%d" % (r[0], r[2]))
@pytest.mark.parametrize("kv_outer", [True, False])
def test_blocked_equals_naive_fp64(row, kv_outer):
    """Same page, section 4.2: blocked and naive agree to rounding (~1e-15)."""
    N, D, causal, printed_max, _ = row
    N, D, causal = int(N), int(D), bool(causal)
    Q, K, V = _normal(N, N, D)
    ref, lse_ref = fa_ref.naive(Q, K, V, 1 / math.sqrt(D), causal)
    got, lse, _, _ = fa_ref.blocked(Q, K, V, 1 / math.sqrt(D), causal, Br=64, Bc=64,
                                    kv_outer=kv_outer)
    err = np.abs(ref - got).max()
    assert err <= 1e-12
    assert err <= 20 * printed_max          # same order as the page's FP64 table
    assert np.abs(lse - lse_ref).max() <= 1e-12


def test_rescale_is_load_bearing():
    """Same page, section 09: with corr forced to 1 the output is wrong."""
    g = kv("rescale_ablation.txt")
    N, D = int(g["N"]), int(g["D"])
    Q, K, V = _normal(N, N, D)
    ref, _ = fa_ref.naive(Q, K, V, 1 / math.sqrt(D), False)
    bad, _, _, _ = fa_ref.blocked(Q, K, V, 1 / math.sqrt(D), False, Br=64, Bc=64,
                                  kv_outer=True, rescale=False)
    err = np.abs(ref - bad)
    assert round(float(err.max()), 3) == float(g["max_abs_err"])
    assert round(float(err.mean()), 4) == float(g["mean_abs_err"])
    good, _, _, _ = fa_ref.blocked(Q, K, V, 1 / math.sqrt(D), False, Br=64, Bc=64, kv_outer=True)
    assert np.abs(ref - good).max() <= 1e-12


def test_causal_block_count():
    """Same page, section 4.5: 2080 of 4096 block pairs at N=4096, block 64."""
    g = kv("causal_block_count.txt")
    N, b = int(g["N"]), int(g["block"])
    z = np.zeros((N, 1))
    _, _, _, vis_c = fa_ref.blocked(z, z, z, 1.0, True, Br=b, Bc=b)
    _, _, _, vis_n = fa_ref.blocked(z, z, z, 1.0, False, Br=b, Bc=b)
    assert vis_n == int(g["pairs_noncausal"])
    assert vis_c == int(g["pairs_causal"])
    T = N // b
    assert vis_c == T * (T + 1) // 2
    assert round(100.0 * (1 - vis_c / vis_n), 1) == float(g["skipped_percent"])


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_visible_values(causal):
    """All-equal scores (mpbf.cn/news/61284, section 5.1 test cases): O_i is the
    mean of the visible v_j and LSE_i = ln(#visible)."""
    N, D = 37, 5
    rng = np.random.default_rng(7)
    Q = np.zeros((N, D)); K = rng.normal(size=(N, D)); V = rng.normal(size=(N, D))
    vis = np.arange(1, N + 1) if causal else np.full(N, N)
    want = np.cumsum(V, 0) / vis[:, None] if causal else np.tile(V.mean(0), (N, 1))
    for o, lse in (fa_ref.naive(Q, K, V, 0.3, causal),
                   fa_ref.blocked(Q, K, V, 0.3, causal, Br=4, Bc=3)[:2]):
        assert np.abs(o[0, 0] - want).max() < 1e-14
        assert np.abs(lse[0, 0] - np.log(vis)).max() < 1e-14


def test_dominant_score_selects_its_value():
    """One score far above the rest: O_i equals that key's value, no overflow."""
    N = D = 16
    rng = np.random.default_rng(3)
    K = np.eye(N)
    perm = rng.permutation(N)
    Q = 800.0 * np.eye(N)[perm]           # row i scores 800 on key perm[i], 0 elsewhere
    V = rng.normal(size=(N, D))
    for o, lse in (fa_ref.naive(Q, K, V, 1.0, False),
                   fa_ref.blocked(Q, K, V, 1.0, False, Br=5, Bc=3)[:2]):
        assert np.all(np.isfinite(o))
        assert np.abs(o[0, 0] - V[perm]).max() < 1e-15
        assert np.abs(lse[0, 0] - 800.0).max() < 1e-12


def test_causal_row_zero_is_v0():
    """Causal mask (CUDA FlashAttention page, section 1): row 0 sees key 0 only."""
    Q, K, V = _normal(11, 9, 6)
    for o, lse in (fa_ref.naive(Q, K, V, 0.4, True),
                   fa_ref.blocked(Q, K, V, 0.4, True, Br=2, Bc=4)[:2]):
        assert np.array_equal(o[0, 0, 0], V[0])
        assert lse[0, 0, 0] == 0.4 * float(Q[0] @ K[0])


@pytest.mark.parametrize("causal", [False, True])
def test_extreme_inputs_stay_finite(causal):
    """fp16 max (65504) and mixed +-1e4 entries (mpbf.cn/news/61284, 5.1):
    the max subtraction keeps O finite and inside the hull of V."""
    N, D = 40, 8
    rng = np.random.default_rng(5)
    Q = rng.choice([-1e4, 1e4, 65504.0, 0.5], size=(N, D))
    K = rng.choice([-1e4, 1e4, 65504.0, -0.5], size=(N, D))
    V = rng.normal(size=(N, D))
    for o, lse in (fa_ref.naive(Q, K, V, 0.125, causal),
                   fa_ref.blocked(Q, K, V, 0.125, causal, Br=8, Bc=16)[:2]):
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        assert np.all(o[0, 0] <= V.max(0) + 1e-12) and np.all(o[0, 0] >= V.min(0) - 1e-12)


def _library_attention(Q, K, V, scale, causal):
    """Direct route through scipy's softmax (no max shift needed at these sizes)."""
    S = scale * (Q @ K.T)
    if causal:
        S = np.where(np.tri(len(Q), dtype=bool), S, -np.inf)
    return scipy.special.softmax(S, axis=1) @ V, scipy.special.logsumexp(S, axis=1)


@pytest.mark.parametrize("N", [1, 2, 3, 17, 127, 128, 129, 255])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(N, D, causal):
    """Any block size gives the same result ('Why FlashAttention ...', 3.2):
    naive, blocked with B_c in {1,2,64,128}, and scipy's softmax agree."""
    rng = np.random.default_rng(1000 * N + D)
    Q, K, V = (rng.normal(size=(N, D)) * 0.3 for _ in range(3))
    scale = 1 / math.sqrt(D)
    want, want_lse = _library_attention(Q, K, V, scale, causal)
    o, lse = fa_ref.naive(Q, K, V, scale, causal)
    assert np.abs(o[0, 0] - want).max() < 1e-13 and np.abs(lse[0, 0] - want_lse).max() < 1e-13
    for bc in (1, 2, 64, 128):
        for br, outer in ((1, True), (64, False), (N, True)):
            ob, lb, _, _ = fa_ref.blocked(Q, K, V, scale, causal, Br=br, Bc=bc, kv_outer=outer)
            assert np.abs(ob[0, 0] - want).max() < 1e-13
            assert np.abs(lb[0, 0] - want_lse).max() < 1e-13


def test_shift_invariance():
    """Adding c to every score of a row leaves O unchanged and adds c to LSE."""
    N, D = 50, 6
    Q, K, V = _normal(9, N, D)
    K2 = K.copy(); K2[:, 0] = 1.0
    Q2 = Q.copy(); Q2[:, 0] += 3.0
    o1, l1 = fa_ref.naive(Q, K2, V, 0.5, True)
    o2, l2 = fa_ref.naive(Q2, K2, V, 0.5, True)
    assert np.abs(o1 - o2).max() < 1e-13
    assert np.abs((l2 - l1) - 1.5).max() < 1e-12


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_16bit_decoding_is_exact(dt):
    """The oracle's binary16 / bfloat16 decoding equals torch's exact upcast,
    including subnormals, infinities' neighbours and signed zero."""
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(2, 3, 33, 8, generator=g) * 4).to(dt)
    special = torch.tensor([0.0, -0.0, 6.0e-8, -6.0e-8, 1e-5, 65504.0, -65504.0, 1.0, -2.5],
                           dtype=torch.float32).to(dt)
    x.view(-1)[: special.numel()] = special
    ks, vs = x.roll(1, 2), x.roll(2, 2)
    from fa_inputs import bits
    o16, l16 = fa_ref.naive(bits(x), bits(ks), bits(vs), 0.2, True,
                            enc="f16" if dt == torch.float16 else "bf16")
    o64, l64 = fa_ref.naive(x.double().numpy(), ks.double().numpy(), vs.double().numpy(), 0.2, True)
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)


def test_rows_entry_matches_full():
    """The selected-rows entry evaluates the same definition row by row."""
    B, H, N, D = 2, 3, 70, 16
    rng = np.random.default_rng(4)
    Q, K, V = (rng.normal(size=(B, H, N, D)) for _ in range(3))
    o, lse = fa_ref.naive(Q, K, V, 0.25, True)
    bh = rng.integers(0, B * H, 40); rows = rng.integers(0, N, 40)
    orow, lrow = fa_ref.naive_rows(Q, K, V, 0.25, True, bh, rows)
    assert np.array_equal(orow, o.reshape(B * H, N, D)[bh, rows])
    assert np.array_equal(lrow, lse.reshape(B * H, N)[bh, rows])


def test_split_merge_worked_row():
    """mpbf.cn/news/61284, section 2.2, as two workers: chunk [1,2] has local
    max 2 and sum 1.368, chunk [3,4] local max 4 and sum 1.368; merged at max 4
    the sum is 1.368 * e^-2 + 1.368 = 1.553 (the split-K reduction of the CUDA
    FlashAttention page, section 7, uses the same merge)."""
    g = kv("worked_row_split.txt")
    scores = [float(x) for x in g["scores"].split()]
    N = len(scores)
    q = np.zeros((N, 1)); q[0, 0] = 1.0
    k = np.array(scores).reshape(N, 1)
    v = np.ones((N, 1))
    _, lse, pm, pl = fa_ref.split_merge(q, k, v, 1.0, chunk=int(g["block_split"]), parts=2)
    dec = int(g["printed_decimals"])
    assert list(pm) == [2.0, 4.0]
    assert round(pl[0], dec) == float(g["block1_sum"]) and round(pl[1], dec) == float(g["block1_sum"])
    merged = pl[0] * math.exp(pm[0] - pm[1]) + pl[1]
    assert round(merged, dec) == float(g["block2_sum"])
    assert abs(lse[0, 0, 0] - (4.0 + math.log(merged))) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("chunk", [1, 7, 64, 128, 1000])
def test_split_merge_equals_naive(causal, chunk):
    """The merged result is the exact attention: it equals the naive form to
    rounding, for any chunk size, including chunks past every visible key."""
    Q, K, V = _normal(77, 300, 32)
    ref, lref = fa_ref.naive(Q, K, V, 0.2, causal)
    got, lgot = fa_ref.split_merge(Q, K, V, 0.2, causal, chunk=chunk)
    assert np.abs(ref - got).max() < 1e-12 and np.abs(lref - lgot).max() < 1e-12


@pytest.mark.parametrize("H,H_kv", [(8, 8), (8, 2), (6, 3), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_attention_on_repeated_kv(H, H_kv, causal):
    """Grouped K/V heads are the same computation as copying each K/V head to
    its H / H_kv query heads (CUDA FlashAttention page, section 7, describes
    the mapping as a way to avoid that copy)."""
    B, N, D = 2, 70, 16
    rng = np.random.default_rng(H * 10 + H_kv)
    q = rng.normal(size=(B, H, N, D)); k = rng.normal(size=(B, H_kv, N, D)); v = rng.normal(size=(B, H_kv, N, D))
    o, lse = fa_ref.naive_gqa(q, k, v, 0.3, causal)
    rep = H // H_kv
    o2, lse2 = fa_ref.naive(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), 0.3, causal)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_gqa_head_mapping_is_grouped_not_strided():
    """Query head h reads K/V head h // (H / H_kv): give each K/V head a
    constant value and read it back through uniform scores."""
    B, H, H_kv, N, D = 1, 6, 2, 5, 4
    q = np.zeros((B, H, N, D)); k = np.zeros((B, H_kv, N, D))
    v = np.stack([np.full((N, D), float(g + 1)) for g in range(H_kv)])[None]
    o, _ = fa_ref.naive_gqa(q, k, v, 1.0)
    for h in range(H):
        assert np.all(o[0, h] == h // (H // H_kv) + 1)
