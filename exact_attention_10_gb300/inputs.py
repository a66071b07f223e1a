"""Seeded synthetic inputs for the attention forward.

This module is shared by the CUDA-path tests, the oracle tests and bench.py.
It holds no attention arithmetic: it only names the workloads and draws their
inputs.

Recipe: Q, K and V are drawn i.i.d. N(0, 1) in float32 on the CPU with
``torch.Generator().manual_seed(seed)``, in the order Q, K, V, each of shape
[B, H, N, D]; for the large-logit stress workload Q and K are then multiplied
by 4 (a power of two, so multiplying before or after rounding gives the same
bits); finally each tensor is rounded to the workload's dtype (round to
nearest even).  This is the input distribution of every workload on the pages
(torch.randn in bf16/fp16, with Q and K amplified 4x in the stability case of
"Building a Verifiable FlashAttention Forward from PyTorch to Triton",
Part 4).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, dtype, scale and input recipe."""

    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str              # "bf16" or "fp16"
    scale: float
    qk_gain: float = 1.0    # Q and K multiplied by this after drawing
    masks: tuple = (False, True)   # causal settings this workload is run with

    @property
    def torch_dtype(self):
        return _TORCH_DTYPE[self.dtype]

    def with_n(self, N: int) -> "Workload":
        return replace(self, N=N, name=f"{self.name}@N{N}")

    def describe(self) -> str:
        gain = f", Q,K x{self.qk_gain:g}" if self.qk_gain != 1.0 else ""
        return (f"B{self.B} H{self.H} N{self.N} D{self.D} {self.dtype}, scale {self.scale:.6g}{gain}")


WORKLOADS = {
    # tiny check, two query tiles
    "tiny_n256": Workload("tiny_n256", 1, 1, 256, 64, "bf16", 1.0 / math.sqrt(64)),
    # medium batch of heads
    "b4h16_n1024": Workload("b4h16_n1024", 4, 16, 1024, 64, "bf16", 1.0 / 8),
    # the N = 4096 comparison scale of the pages (B*H = 32, D = 64)
    "b2h16_n4096": Workload("b2h16_n4096", 2, 16, 4096, 64, "bf16", 1.0 / 8),
    # ragged N (not a tile multiple), D = 128, fp16, large logits
    "ragged_n3000_d128_fp16": Workload("ragged_n3000_d128_fp16", 2, 8, 3000, 128, "fp16",
                                       1.0 / math.sqrt(128), qk_gain=4.0),
    # long context: causal at N = 32768; non-causal is run at N = 16384
    "long_n32768_d128": Workload("long_n32768_d128", 1, 32, 32768, 128, "bf16", 1.0 / math.sqrt(128),
                                 masks=(True,)),
    "long_n16384_d128": Workload("long_n16384_d128", 1, 32, 16384, 128, "bf16", 1.0 / math.sqrt(128),
                                 masks=(False,)),
}


def make_qkv(w: Workload, seed: int = 0, device: str | torch.device = "cpu"):
    """Draw (Q, K, V) for workload ``w`` with ``seed``; returns contiguous [B,H,N,D] tensors."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (w.B, w.H, w.N, w.D)
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if which in ("q", "k") and w.qk_gain != 1.0:
            x.mul_(w.qk_gain)
        out.append(x.to(w.torch_dtype).to(device).contiguous())
    return tuple(out)


def make_custom(B: int, H: int, N: int, D: int, dtype: str, seed: int = 0, qk_gain: float = 1.0,
                device: str | torch.device = "cpu"):
    """Same recipe for an arbitrary shape (used by the edge-case tests)."""
    w = Workload(f"custom_b{B}h{H}n{N}d{D}", B, H, N, D, dtype, 1.0 / math.sqrt(D), qk_gain)
    return make_qkv(w, seed, device)
