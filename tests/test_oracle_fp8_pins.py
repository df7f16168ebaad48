"""Pins of the oracle's FP8 (OCP E4M3) decoding and per-block dequantization.

The FP8 path computes attention of dequantized inputs: value = E4M3(x) times
the fp32 scale of its 128-row block ("CUDA FlashAttention: from online
softmax to the long-sequence IO limit", section 2: 8-bit inputs need a
per-tensor or per-block scale).  The oracle decodes the bytes itself; these
tests tie that decoder to torch's float8_e4m3fn and to the format's
definition, and check the block bookkeeping.
"""
import numpy as np
import pytest
import torch

import fa_inputs
from oracle import fa_ref


def test_every_e4m3_pattern_matches_torch():
    bytes_ = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = bytes_.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([fa_ref.decode_e4m3(b) for b in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("byte,value", [(0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0x01, 2.0 ** -9),
                                        (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x3C, 1.5), (0x40, 2.0)])
def test_e4m3_definition(byte, value):
    assert fa_ref.decode_e4m3(byte) == value


def test_dequant_applies_each_blocks_scale():
    rng = np.random.default_rng(0)
    B, H, N, D, blk = 2, 3, 300, 16, 128          # 3 blocks per head, the last one ragged
    x = rng.integers(0, 256, size=(B, H, N, D), dtype=np.uint8)
    x[(x & 0x7F) == 0x7F] = 0x3F                   # no NaN patterns
    sc = rng.uniform(0.01, 2.0, size=(B, H, 3)).astype(np.float32)
    got = fa_ref.dequant_e4m3(x, sc, blk)
    dec = torch.from_numpy(x).view(torch.float8_e4m3fn).double().numpy()
    want = dec * np.repeat(sc.astype(np.float64), blk, axis=2)[:, :, :N, None]
    assert np.array_equal(got, want)


def test_block_quantization_error_bound():
    w = fa_inputs.Workload("fp8", 1, 2, 300, 128, False, "bf16")
    (q8, k8, v8), (qs, ks, vs) = fa_inputs.make_qkv_fp8(w, seed=3)
    g = torch.Generator().manual_seed(3)
    q = torch.randn((1, 2, 300, 128), generator=g).double().numpy()
    deq = fa_ref.dequant_e4m3(q8.numpy(), qs.numpy())
    s = np.repeat(qs.double().numpy(), 128, axis=2)[:, :, :300, None]
    # round to nearest: half an ulp, 2^-4 relative for normals, 2^-10 * scale below 2^-6 * scale
    bound = np.maximum(np.abs(q) * 2.0 ** -4, s * 2.0 ** -10)
    assert np.all(np.abs(deq - q) <= bound * (1 + 1e-12))
    # the block maximum maps to 448 exactly
    assert np.allclose(np.abs(deq).reshape(1, 2, -1).max(axis=-1), np.abs(q).reshape(1, 2, -1).max(axis=-1),
                       rtol=2.0 ** -4)
