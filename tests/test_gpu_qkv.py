"""Fused QKV projection with the KV append in its epilogue (mg_qkv_append)
against the fp64 oracle: hidden size 6656 -> 32 query heads and 2 key / 2
value heads of 128 ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
section 01).

Reading of the tolerance: the kernel multiplies bf16 values exactly and
accumulates 6656 products in fp32, then rounds once to bf16.  So every output
lies within half a bf16 ulp of the fp64 value plus the fp32 accumulation bound
gamma_6656 |x| |W|^T, and differs from the correctly rounded value only where
the fp64 value sits within that bound of a rounding midpoint (rare: checked
as a fraction).  The cache is checked bit for bit: it must hold exactly the
key / value rows the kernel produced, placed as the oracle's append places
them."""
import numpy as np
import pytest
import torch

from gpu_util import check_err
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


@pytest.fixture(scope="module")
def weights():
    # sigma 1/64: outputs of sigma ~1.3
    return synth.scaled(synth.randn_bf16((orc.QKV_FEATURES, orc.HIDDEN), 71), 1.0 / 64)


def check_values(y_gpu, x_rows, w, what):
    """y_gpu: bf16 [rows][4608] (cpu); x_rows: bf16 [rows][6656]."""
    ref = orc.qkv_project(x_rows, w)
    bound = orc.FP32_GAMMA_HIDDEN * orc.qkv_abs_bound(x_rows, w)
    got = y_gpu.float().double().numpy()
    ax = np.abs(ref)
    _, e = np.frexp(ax)
    half_ulp = np.where(ax > 0, np.ldexp(1.0, e - 9), 0.0)
    diff = np.abs(got - ref)
    assert (diff <= half_ulp + bound).all(), f"{what}: worst excess {(diff - half_ulp - bound).max():.3e}"
    # Where the fp64 value lies within the accumulation error of a rounding
    # midpoint the kernel may round the other way: on B300 about 0.4 % of
    # these outputs do (an accumulation error near 1e-5 against a bf16 ulp of
    # 2^-7 at |y| ~ 1); a wrong operand, index or dropped K slice would move
    # most of them.
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    off = np.mean(got != rounded)
    assert off < 1e-2, f"{what}: {off:.2e} of the outputs are not the correctly rounded value"
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 4e-3, f"{what}: rel-L2 {rel:.3e}"


def run(mg, kind, cache, pos0, x, w, with_kv_out=True):
    B, n = x.shape[0], x.shape[1]
    lay = mg.make_layer(kind)
    q = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, n, 2, 128), dtype=torch.bfloat16, device="cuda") if with_kv_out else None
    v = torch.empty_like(k) if with_kv_out else None
    ws = mg.qkv_workspace(B, n)
    err = mg.error_word()
    mg.mg_qkv_append(lay, cache, torch.tensor(pos0, dtype=torch.int32, device="cuda"),
                     x.cuda().contiguous(), w.cuda().contiguous(), q, ws, err, k_out=k, v_out=v)
    torch.cuda.synchronize()
    return q, k, v, err


def expected_cache(kind, cache, pos0, k, v):
    """Oracle replay of the append of the kernel's own rows onto the
    cache's previous contents (uint16 bits per sequence)."""
    out = []
    for b, p0 in enumerate(pos0):
        kc = cache[0][b].cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        vc = cache[1][b].cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        orc.cache_append(orc.LOCAL if kind == 0 else orc.GLOBAL, kc, vc, p0, k[b].cpu(), v[b].cpu())
        out.append((kc, vc))
    return out


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kind,B,n,pos0", [
    (1, 2, 300, [0, 1000]),          # 600 tokens: 5 row tiles (ragged), one pass per CTA
    (0, 3, 1, [5000, 2047, 10]),     # decode: the K range split 8 ways, then the reduction
    (1, 4, 40, [7, 0, 300, 129]),    # 160 tokens: split 4 ways
    (0, 1, 2100, [100]),             # more than 2048 tokens into the ring: the last 2048 stay
])
def test_qkv_append_against_oracle(mg, weights, kind, B, n, pos0):
    x = synth.randn_bf16((B, n, orc.HIDDEN), 72 + n)
    cap = max(pos0) + n
    cache = mg.KVCache(kind, B, cap)
    cache.k.normal_()  # previous contents the append must leave where it does not write
    cache.v.normal_()
    before = (cache.k.clone(), cache.v.clone())
    q, k, v, err = run(mg, kind, cache, pos0, x, weights)
    check_err(err)
    y = torch.cat([q.reshape(B * n, -1), k.reshape(B * n, -1), v.reshape(B * n, -1)], dim=1).cpu()
    rows = np.arange(B * n)
    if B * n > 400:  # the fp64 product of every row would take long: a sample with both ends
        rows = np.unique(np.concatenate([rows[:96], rows[-96:], rows[::37]]))
    check_values(y[rows], x.reshape(B * n, -1)[rows], weights, f"kind {kind} B {B} n {n}")
    exp = expected_cache(kind, before, pos0, k, v)
    for b in range(B):
        assert np.array_equal(bits(cache.k[b]), exp[b][0]), f"K cache of sequence {b}"
        assert np.array_equal(bits(cache.v[b]), exp[b][1]), f"V cache of sequence {b}"


def test_qkv_append_paged_and_without_kv_out(mg, weights):
    # a paged global cache (pages handed out in shuffled order), and the same
    # call without k_out / v_out: the stored rows are identical
    B, n, ps = 2, 200, 256
    pos0 = [100, 700]
    x = synth.randn_bf16((B, n, orc.HIDDEN), 73)
    cap = 1024
    paged = mg.PagedKVCache(B, cap, num_pages=8, page_size=ps)
    paged.table.copy_(torch.tensor([[5, 2, 7, 0], [3, 6, 1, 4]], dtype=torch.int32))
    lin = mg.KVCache(1, B, cap)
    q, k, v, err = run(mg, 1, lin, pos0, x, weights)
    check_err(err)
    q2, _, _, err2 = run(mg, 1, paged, pos0, x, weights, with_kv_out=False)
    check_err(err2)
    assert torch.equal(q, q2)
    for b, p0 in enumerate(pos0):
        kp, vp = paged.linear(b, p0 + n)
        assert torch.equal(kp[:, p0:], lin.k[b, :, p0:p0 + n])
        assert torch.equal(vp[:, p0:], lin.v[b, :, p0:p0 + n])
        assert torch.equal(lin.k[b, :, p0:p0 + n].transpose(0, 1), k[b])


def test_qkv_append_flags_a_bad_position(mg, weights):
    B, n = 2, 3
    x = synth.randn_bf16((B, n, orc.HIDDEN), 74)
    cache = mg.KVCache(1, B, 64)
    q, k, v, err = run(mg, 1, cache, [-1, 61], x, weights)  # 61 + 2 = 63 < 64: fine
    assert int(err.item()) == mg.DERR_POSITION
    assert not cache.k[0].any()  # nothing stored for the rejected sequence
    assert torch.equal(cache.k[1, :, 61:64].transpose(0, 1), k[1])
