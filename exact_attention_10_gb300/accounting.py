"""FLOP and byte accounting for the attention forward (host logic for bench.py).

Conventions are the pages':
  * useful FLOPs = 4*B*H*N^2*D (two N x N x D matmuls), halved for causal
    ("FlashAttention 2 from PyTorch to Triton", Step 4: the benchmark;
    "How to profile and optimise kernels", 137.4 G at B*H=32, N=4096, D=64);
  * fused HBM traffic = Q, K, V read once and O written once, 8*N*d bytes per
    head in a 16-bit type ("A09 - Advanced Triton & FlashAttention",
    2. First Principles), plus the fp32 LSE row this library also writes;
  * unfused traffic adds 4 passes over the 2*N^2-byte score matrix, so the
    ratio unfused/fused is 1 + N/d (same section).
"""
from __future__ import annotations


def flops(B: int, H: int, N: int, D: int, causal: bool) -> float:
    """The pages' FLOP count: 4*B*H*N^2*D, half of it when causal."""
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


def flops_causal_exact(B: int, H: int, N: int, D: int) -> float:
    """Exact causal count: 4*B*H*D * N(N+1)/2 (the diagonal included)."""
    return 4.0 * B * H * D * N * (N + 1) / 2


def fused_bytes(B: int, H: int, N: int, D: int, elem_bytes: int = 2, with_lse: bool = True) -> int:
    """Algorithmic HBM bytes of one forward: read Q, K, V, write O (and the fp32 LSE)."""
    b = 4 * B * H * N * D * elem_bytes
    if with_lse:
        b += 4 * B * H * N
    return b


def unfused_bytes_per_head(N: int, D: int, elem_bytes: int = 2) -> int:
    """Three-kernel attention: Q, K, V, O plus four passes over the N x N scores."""
    return 4 * N * D * elem_bytes + 4 * (elem_bytes * N * N)


def unfused_ratio(N: int, D: int) -> float:
    return 1.0 + N / D


def l2_operand_bytes(B: int, H: int, N: int, D: int, causal: bool, cta_rows: int = 256, bn: int = 128,
                     elem_bytes: int = 2) -> int:
    """Bytes of K and V the kernel's CTA tiles fetch through L2 (each CTA tile of
    ``cta_rows`` queries reads its head's K/V once, up to the diagonal when causal)."""
    tiles = -(-N // cta_rows)
    kv_tiles_total = 0
    for t in range(tiles):
        if causal:
            last = min(t * cta_rows + cta_rows - 1, N - 1)
            kv_tiles_total += last // bn + 1
        else:
            kv_tiles_total += -(-N // bn)
    return B * H * kv_tiles_total * 2 * bn * D * elem_bytes
