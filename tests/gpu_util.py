"""Shared pieces of the GPU parity tests: tolerances, comparison, cache
construction through the library, and the oracle's per-sequence calls."""
import numpy as np
import torch

from oracle import oracle as orc

# Parity bar for bf16 in / fp32 accumulate against the fp64 oracle:
#   per element  |o_gpu - o_ref| <= MAX_ABS + half an ulp of bf16 at |o_ref|
#   overall      ||o_gpu - o_ref||_2 / ||o_ref||_2 <= REL_L2
# The output is bf16, so no result can be closer to the exact value than
# half a bf16 ulp (2^-8 relative); from |o| >= 4 that alone exceeds 1e-2.
# MAX_ABS therefore bounds the arithmetic error on top of the output format.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (bf16 keeps 8 significant bits)."""
    ax = np.abs(x)
    _, e = np.frexp(ax)  # ax = f * 2^e, f in [0.5, 1)
    return np.where(ax > 0, np.ldexp(1.0, e - 9), 0.0)


def compare(o_gpu, o_ref, what=""):
    """o_gpu: bf16 tensor (any device); o_ref: float64 array of the same shape.
    Returns (raw max-abs, excess over the bf16 half-ulp, rel-L2)."""
    og = o_gpu.detach().float().cpu().double().numpy()
    ref = np.asarray(o_ref, dtype=np.float64)
    assert og.shape == ref.shape, (og.shape, ref.shape)
    assert np.isfinite(og).all(), f"{what}: non-finite output"
    diff = np.abs(og - ref)
    raw = diff.max()
    excess = (diff - half_ulp_bf16(ref)).max()
    rel = np.linalg.norm(og - ref) / max(np.linalg.norm(ref), 1e-30)
    assert excess <= MAX_ABS and rel <= REL_L2, (
        f"{what}: max-abs {raw:.3e} (beyond bf16 half-ulp {excess:.3e}) rel-L2 {rel:.3e}")
    return raw, excess, rel


def oracle_kind(kind):
    return orc.LOCAL if kind == 0 else orc.GLOBAL


def cache_expected(kind, slots, k_hist, v_hist, appends):
    """Oracle replay of appends [(pos0, n), ...] of one sequence -> (k, v) uint16."""
    kc = np.zeros((2, slots, 128), np.uint16)
    vc = np.zeros((2, slots, 128), np.uint16)
    for pos0, n in appends:
        orc.cache_append(oracle_kind(kind), kc, vc, pos0, k_hist[pos0:pos0 + n], v_hist[pos0:pos0 + n])
    return kc, vc


def bits_of(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_err(err, expect=0):
    v = int(err.item())
    assert v == expect, f"device error word {v:#x}, expected {expect:#x}"
