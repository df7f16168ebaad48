"""bench.py's statistics on CPU: rounding to the output type (the
quantisation floor of the accuracy report), the error statistics, and the
median of group means."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_round_to_matches_torch_casts_of_float32_values():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * 4, torch.randn(2000, generator=g) * 1e-3])
    for dtype, td in (("fp16", torch.float16), ("bf16", torch.bfloat16)):
        want = x.to(td).double().numpy()
        got = bench.round_to(x.double().numpy(), dtype)
        assert np.array_equal(got, want), dtype


def test_round_to_ties_go_to_even():
    assert bench.round_to(np.array([1 + 2.0 ** -11]), "fp16")[0] == 1.0
    assert bench.round_to(np.array([1 + 3 * 2.0 ** -11]), "fp16")[0] == 1 + 2.0 ** -9
    assert bench.round_to(np.array([1 + 2.0 ** -8]), "bf16")[0] == 1.0
    assert bench.round_to(np.array([1 + 3 * 2.0 ** -8]), "bf16")[0] == 1 + 2.0 ** -6


def test_accuracy_stats_values():
    o_ref = np.array([[1.0, 2.0], [3.0, 0.5]])
    o = o_ref + np.array([[0.0, 1e-3], [-2e-3, 0.0]])
    s = bench.accuracy_stats(o, np.array([0.1, 0.2]), o_ref, np.array([0.1, 0.2005]), "fp16")
    assert abs(s["max_abs_o"] - 2e-3) < 1e-15 and abs(s["rms_o"] - np.sqrt(5e-6 / 4)) < 1e-15
    assert abs(s["max_abs_lse"] - 5e-4) < 1e-12 and s["quant_floor_o"] == 0.0 and s["elements"] == 4
    assert abs(s["rel_l2_o"] - np.sqrt(5e-6) / np.linalg.norm(o_ref)) < 1e-15


def test_group_median_of_means():
    xs = [float(g) for g in (5, 1, 3, 7, 2, 6, 4) for _ in range(3)] + [100.0]
    assert bench.group_median(xs) == 4.0
    assert bench.group_median([1.0] * 6) is None
