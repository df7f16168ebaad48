"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and names shapes; it holds none of the
attention arithmetic.  The tests, the smoke check and the bench take their
inputs from here, so the CUDA path and the FP64 oracle see the same values.

Recipe (every workload): one CPU ``torch.Generator`` seeded with ``seed``
(default 0) draws ``randn([B,H,N,D], float32)`` for Q, then K, then V; the
"peaky" stress workload multiplies Q and K by its ``qk_std`` of 3; the three
tensors are then rounded to the workload's 16-bit dtype (round to nearest
even).  The oracle decodes those rounded values exactly.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    causal: bool
    dtype: str          # "fp16" or "bf16"
    qk_std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def flops(self) -> float:
        """Attention forward FLOPs: 4*B*H*N^2*D, or half of it when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.D
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Q, K, V read once, O written once (2 bytes each), LSE once (4 bytes)."""
        elems = self.B * self.H * self.N * self.D
        return 4 * elems * 2 + self.B * self.H * self.N * 4

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads the method is measured and checked on.
WORKLOADS = {
    "tiny_fp16_b1h2n256d64": Workload("tiny_fp16_b1h2n256d64", 1, 2, 256, 64, False, "fp16"),
    "noncausal_fp16_b1h32n4096d64": Workload("noncausal_fp16_b1h32n4096d64", 1, 32, 4096, 64, False, "fp16"),
    "peaky_causal_bf16_b2h16n16384d128": Workload("peaky_causal_bf16_b2h16n16384d128", 2, 16, 16384, 128,
                                                  True, "bf16", qk_std=3.0),
    "ragged_causal_bf16_b1h8n32749d128": Workload("ragged_causal_bf16_b1h8n32749d128", 1, 8, 32749, 128,
                                                  True, "bf16"),
}
# One long head: too few query blocks to fill the GPU, where splitting the keys pays.
WORKLOADS["longhead_causal_bf16_b1h1n32768d128"] = Workload("longhead_causal_bf16_b1h1n32768d128", 1, 1, 32768, 128,
                                                             True, "bf16")
for _n in (512, 1024, 2048, 4096, 8192):
    _w = Workload("causal_fp16_b1h32n%dd128" % _n, 1, 32, _n, 128, True, "fp16")
    WORKLOADS[_w.name] = _w


def make_qkv(w: Workload, seed: int = 0):
    """Q, K, V as CPU tensors of the workload's dtype, drawn as the recipe says."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (w.B, w.H, w.N, w.D)
    out = []
    for i in range(3):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if i < 2 and w.qk_std != 1.0:
            t.mul_(w.qk_std)
        out.append(t.to(w.torch_dtype))
    return tuple(out)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU fp16/bf16 tensor, as a uint16 numpy array."""
    assert t.dtype in (torch.float16, torch.bfloat16) and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def enc(w_or_dtype) -> str:
    """Oracle encoding name for a workload or a torch dtype."""
    d = w_or_dtype.torch_dtype if isinstance(w_or_dtype, Workload) else w_or_dtype
    return "f16" if d == torch.float16 else "bf16"


E4M3_MAX = 448.0


def quantize_e4m3_blocks(x, block_rows=128):
    """Per-block FP8 quantization of x [B,H,N,D] (float): for every block of
    block_rows rows of a head, scale = amax / 448 (1 for an all-zero block) and
    q = E4M3(x / scale), rounded to nearest even by torch's float8_e4m3fn cast.
    Returns (q as uint8 bit patterns [B,H,N,D], scales float32 [B,H,nb])."""
    B, H, N, D = x.shape
    nb = (N + block_rows - 1) // block_rows
    xf = x.float()
    pad = nb * block_rows - N
    xp = torch.nn.functional.pad(xf, (0, 0, 0, pad)) if pad else xf
    amax = xp.reshape(B, H, nb, block_rows * D).abs().amax(dim=-1)
    scales = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
    rows_scale = scales.repeat_interleave(block_rows, dim=2)[:, :, :N, None]
    q8 = (xf / rows_scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8), scales


def make_qkv_fp8(w, seed=0):
    """N(0,1) Q, K, V of workload w (drawn as in make_qkv, before any cast),
    quantized per 128-row block: ((q8, k8, v8) uint8 [B,H,N,D], (qs, ks, vs))."""
    g = torch.Generator().manual_seed(seed)
    shape = (w.B, w.H, w.N, w.D)
    q = torch.randn(shape, generator=g) * w.qk_std
    k = torch.randn(shape, generator=g) * w.qk_std
    v = torch.randn(shape, generator=g)
    out = [quantize_e4m3_blocks(t) for t in (q, k, v)]
    return tuple(o[0] for o in out), tuple(o[1] for o in out)
