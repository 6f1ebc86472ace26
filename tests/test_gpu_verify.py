"""Speculative verify (a block of up to 16 draft tokens in one pass, causal
inside the block) against the oracle, and against 16 sequential GPU decodes."""
import pytest
import torch

from gpu_util import check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def build_cache(mg, kind, k, v, p0s, capacity):
    """Cache holding positions < p0[b] of each sequence (ring: the last 2048)."""
    B = k.shape[0]
    cache = mg.KVCache(kind, B, capacity)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    for b, p0 in enumerate(p0s):
        if p0 == 0:
            continue
        # append sequence b alone: other sequences get a no-op-sized call
        lo = max(0, p0 - 2048) if kind == 0 else 0
        n = p0 - lo
        pos = torch.tensor([lo] * B, dtype=torch.int32, device="cuda")
        kn = k[:, lo:lo + n].clone()
        vn = v[:, lo:lo + n].clone()
        one = mg.KVCache(kind, 1, capacity)
        mg.mg_kv_append(lay, one, pos[:1], kn[b:b + 1].cuda().contiguous(),
                        vn[b:b + 1].cuda().contiguous(), err)
        cache.k[b].copy_(one.k[0])
        cache.v[b].copy_(one.v[0])
    torch.cuda.synchronize()
    check_err(err)
    return cache


def run_verify(mg, kind, cache, p0s, q, kn, vn, max_len):
    lay = mg.make_layer(kind)
    B, n = q.shape[0], q.shape[1]
    ws = mg.workspace(mg.OP_VERIFY, lay, B, n, max_len)
    o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    mg.mg_attn_verify(lay, cache, torch.tensor(p0s, dtype=torch.int32, device="cuda"), max_len,
                      q.cuda().contiguous(), kn.cuda().contiguous(), vn.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    return o, err


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("p0s,n", [([0, 100], 16), ([2100, 1], 16), ([5000, 130], 5),
                                   ([2032, 2048], 16), ([700, 300], 1),
                                   # blocks that wrap the ring inside themselves, a second
                                   # group of 3 tokens, three sequences
                                   ([2040, 4090, 9], 11), ([6139, 31], 13), ([4095, 2047], 2),
                                   # eight sequences: local clusters of 4 CTAs walking
                                   # their ring pieces in rounds, ragged token groups
                                   ([3, 130, 2047, 2048, 2100, 4095, 5000, 10], 5),
                                   ([600, 1, 2030, 3000, 4096, 2049, 129, 7000], 13)])
def test_verify_against_oracle(mg, kind, p0s, n):
    B = len(p0s)
    T = max(p0s) + n
    li = 2 if kind == 0 else 3
    k, v = synth.history(B, T, 11, li)
    q = synth.queries(B, n, 11, li)
    cache = build_cache(mg, kind, k, v, p0s, capacity=T)
    kn = torch.stack([k[b, p:p + n] for b, p in enumerate(p0s)])
    vn = torch.stack([v[b, p:p + n] for b, p in enumerate(p0s)])
    o, err = run_verify(mg, kind, cache, p0s, q, kn, vn, max_len=T)
    check_err(err)
    lay = orc.layer(oracle_kind(kind))
    for b, p0 in enumerate(p0s):
        ref = orc.attention(lay, k[b, :p0 + n], v[b, :p0 + n], list(range(p0, p0 + n)), q[b])
        compare(o[b], ref, f"kind {kind} b {b} p0 {p0} n {n}")


@pytest.mark.parametrize("kind", [0, 1])
def test_verify_equals_sequential_decodes(mg, kind):
    p0, n = 3000, 16
    T = p0 + n
    li = 2 if kind == 0 else 3
    k, v = synth.history(1, T, 12, li)
    q = synth.queries(1, n, 12, li)
    cache = build_cache(mg, kind, k, v, [p0], capacity=T)
    o_blk, err = run_verify(mg, kind, cache, [p0], q, k[:, p0:], v[:, p0:], max_len=T)
    check_err(err)
    lay = mg.make_layer(kind)
    ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, T)
    o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
    for i in range(n):
        pos = torch.tensor([p0 + i], dtype=torch.int32, device="cuda")
        mg.mg_kv_append(lay, cache, pos, kd[:, p0 + i:p0 + i + 1].contiguous(),
                        vd[:, p0 + i:p0 + i + 1].contiguous(), err)
        mg.mg_attn_decode(lay, cache, pos, T, qd[:, i].contiguous(), o, ws, err)
        # both are within the oracle tolerance; against each other allow twice it
        d = (o[0].float() - o_blk[0, i].float()).abs().max().item()
        assert d <= 2e-2, f"step {i}: verify vs decode differ by {d}"
    torch.cuda.synchronize()
    check_err(err)
