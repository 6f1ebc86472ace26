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


# ---------------------------------------------------------------------------
# Peaked inputs: the same N(0, 1) draws, reshaped so that softmax rows become
# sharp.  These only scale or overwrite input values; they hold no attention
# arithmetic.

# Dimension the sink construction uses.  Its RoPE partner is SINK_DIM + 64;
# dimension 63 has the lowest rotary frequency, so a key there keeps its
# direction across a 2048-token window.
SINK_DIM = 63
SINK_Q = 8.0     # value written into every query at SINK_DIM
SINK_K = 64.0    # value of a sink key at SINK_DIM (all its other dims are 0)


def scaled(x: torch.Tensor, factor: float) -> torch.Tensor:
    """x * factor, rounded once to bf16 (round to nearest even)."""
    return (x.float() * float(factor)).to(torch.bfloat16)


def sink_queries(q: torch.Tensor) -> torch.Tensor:
    """Queries with dimension SINK_DIM set to SINK_Q and its RoPE partner to 0
    (every head, every token); the other dimensions are kept."""
    q = q.clone()
    q[..., SINK_DIM] = SINK_Q
    q[..., SINK_DIM + 64] = 0.0
    return q


def plant_sinks(k: torch.Tensor, positions, seq=None, values=None) -> torch.Tensor:
    """Key history [B][T][2][128] with the rows at `positions` (of every
    sequence, or of sequence `seq`) replaced by value * e_SINK_DIM in both KV
    heads (value SINK_K unless `values` gives one per position).  Against
    sink_queries such a key scores SINK_Q * value / sqrt(128) before rotation
    (about 45 for SINK_K), while ordinary keys score N(0, ~1.5)."""
    k = k.clone()
    rows = k if seq is None else k[seq:seq + 1]
    for n, p in enumerate(positions):
        rows[:, p] = 0.0
        rows[:, p, :, SINK_DIM] = SINK_K if values is None else float(values[n])
    return k
