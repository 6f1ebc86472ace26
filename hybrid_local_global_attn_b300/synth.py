"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

Holds no attention arithmetic: only how random bf16 tensors are drawn.
Recipe: torch's CPU (or CUDA) Philox generator seeded per tensor, fp32
N(0, 1) samples rounded to bf16 (round to nearest even).  A tensor's seed is
``seed * 1000 + layer * 10 + which`` with which = 0 (q), 1 (k), 2 (v).
"""
import torch

Q, K, V = 0, 1, 2


def sub_seed(seed: int, layer: int, which: int) -> int:
    return int(seed) * 1000 + int(layer) * 10 + int(which)


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    return x.to(torch.bfloat16)


def history(batch: int, T: int, seed: int, layer: int, device="cpu"):
    """K and V histories [batch][T][2][128] of one layer."""
    k = randn_bf16((batch, T, 2, 128), sub_seed(seed, layer, K), device)
    v = randn_bf16((batch, T, 2, 128), sub_seed(seed, layer, V), device)
    return k, v


def queries(batch: int, n: int, seed: int, layer: int, device="cpu"):
    """Queries [batch][n][32][128] of one layer."""
    return randn_bf16((batch, n, 32, 128), sub_seed(seed, layer, Q), device)
