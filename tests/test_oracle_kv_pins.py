"""Pins of the oracle's queries-against-a-KV-sequence form (fa_ref_naive_kv).

It must agree with the already pinned square forms where the shapes meet, and
with a brute-force softmax over an explicitly built mask on tiny shapes:
* Nq = Nk reduces it to the square definition (fa_ref_naive / _gqa);
* query i of Nq is the token at position i + Nk - Nq: under the causal mask it
  equals row i + Nk - Nq of the square problem over all Nk tokens;
* a single query (decode) sees every key, with or without the mask.
"""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import fa_ref


def _rand(shape, seed):
    return np.random.default_rng(seed).normal(size=shape)


@pytest.mark.parametrize("causal", [False, True])
def test_square_case_is_the_square_oracle(causal):
    q, k, v = (_rand((2, 4, 37, 16), s) for s in (1, 2, 3))
    a = fa_ref.naive_kv(q, k, v, 0.3, causal)
    b = fa_ref.naive(q, k, v, 0.3, causal)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    kg, vg = k[:, :2], v[:, :2]
    a = fa_ref.naive_kv(q, kg, vg, 0.3, causal)
    b = fa_ref.naive_gqa(q, kg, vg, 0.3, causal)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("nq", [1, 3, 17])
def test_trailing_queries_are_the_last_rows_of_the_square_problem(nq):
    nk = 40
    qfull, k, v = (_rand((1, 2, nk, 8), s) for s in (4, 5, 6))
    o_sq, l_sq = fa_ref.naive(qfull, k, v, 0.5, True)
    o, l = fa_ref.naive_kv(np.ascontiguousarray(qfull[:, :, nk - nq:]), k, v, 0.5, True)
    assert np.abs(o - o_sq[:, :, nk - nq:]).max() <= 1e-13
    assert np.abs(l - l_sq[:, :, nk - nq:]).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_with_an_explicit_mask(causal):
    B, H, H_kv, Nq, Nk, D = 1, 4, 2, 5, 11, 6
    q, k, v = _rand((B, H, Nq, D), 7), _rand((B, H_kv, Nk, D), 8), _rand((B, H_kv, Nk, D), 9)
    o, l = fa_ref.naive_kv(q, k, v, 0.7, causal)
    for h in range(H):
        kk, vv = k[0, h // 2], v[0, h // 2]
        s = 0.7 * q[0, h] @ kk.T
        if causal:
            s = np.where(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq), s, -np.inf)
        assert np.abs(o[0, h] - softmax(s, axis=1) @ vv).max() <= 1e-13
        assert np.abs(l[0, h] - logsumexp(s, axis=1)).max() <= 1e-13


def test_single_query_sees_every_key():
    q, k, v = _rand((2, 8, 1, 32), 10), _rand((2, 2, 300, 32), 11), _rand((2, 2, 300, 32), 12)
    a = fa_ref.naive_kv(q, k, v, 0.2, True)
    b = fa_ref.naive_kv(q, k, v, 0.2, False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
