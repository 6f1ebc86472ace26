"""Speculative commit: after a verify pass the caller keeps the first count[b]
tokens of each sequence's block; the cache must then hold exactly the linear
history of kept tokens ("Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析",
"第三招：D-Flash投机解码实现3倍提速").  Caches are compared bit for bit with the
oracle's, outputs of later verify passes and decodes against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import bits_of, check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

DERR_COUNT = 4


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def oracle_cache(kind, slots, k_hist, v_hist, upto):
    kc = np.zeros((2, slots, 128), np.uint16)
    vc = np.zeros((2, slots, 128), np.uint16)
    if upto:
        orc.cache_append(oracle_kind(kind), kc, vc, 0, k_hist[:upto], v_hist[:upto])
    return kc, vc


def gpu_cache(mg, kind, B, slots, k_hist, v_hist, p0s):
    """Cache of every sequence b holding its positions < p0s[b]."""
    cache = mg.KVCache(kind, B, slots)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    for b, p0 in enumerate(p0s):
        if p0 == 0:
            continue
        one = mg.KVCache(kind, 1, slots)
        pos = torch.zeros(1, dtype=torch.int32, device="cuda")
        mg.mg_kv_append(lay, one, pos, k_hist[b:b + 1, :p0].cuda().contiguous(),
                        v_hist[b:b + 1, :p0].cuda().contiguous(), err)
        cache.k[b].copy_(one.k[0])
        cache.v[b].copy_(one.v[0])
    torch.cuda.synchronize()
    check_err(err)
    return cache


@pytest.mark.parametrize("kind", [0, 1])
def test_commit_cache_bit_exact(mg, kind):
    # Four sequences, block of 16: blocks that cross the ring wrap, a first
    # block at position 0, and counts 0, 16 and partial.
    p0s, counts, n = [2040, 4090, 0, 6000], [5, 16, 0, 11], 16
    B, T = len(p0s), max(p0s) + n
    slots = 2048 if kind == 0 else T
    k, v = synth.history(B, T, 31, 2 if kind == 0 else 3)
    jk, jv = synth.history(B, n, 32, 2 if kind == 0 else 3)  # rejected drafts
    blk_k = torch.stack([torch.cat([k[b, p:p + c], jk[b, c:]]) for b, (p, c) in
                         enumerate(zip(p0s, counts))])
    blk_v = torch.stack([torch.cat([v[b, p:p + c], jv[b, c:]]) for b, (p, c) in
                         enumerate(zip(p0s, counts))])
    cache = gpu_cache(mg, kind, B, slots, k, v, p0s)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    pos0 = torch.tensor(p0s, dtype=torch.int32, device="cuda")
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    mg.mg_kv_commit(lay, cache, pos0, cnt, blk_k.cuda().contiguous(), blk_v.cuda().contiguous(),
                    err, pos_next=nxt)
    torch.cuda.synchronize()
    check_err(err)
    assert nxt.tolist() == [p + c for p, c in zip(p0s, counts)]
    for b in range(B):
        kc, vc = oracle_cache(kind, slots, k[b], v[b], p0s[b])
        orc.cache_commit(oracle_kind(kind), kc, vc, p0s[b], counts[b], blk_k[b], blk_v[b])
        assert np.array_equal(bits_of(cache.k[b]), kc), f"K cache of sequence {b}"
        assert np.array_equal(bits_of(cache.v[b]), vc), f"V cache of sequence {b}"


def test_commit_count_out_of_range_skips_that_sequence(mg):
    # The kernel checks the count (no invalid access is made): sequence 1
    # asks for 17 of 16 tokens and is left as it was, flagged; sequence 0
    # is committed.
    kind, n, p0s = 0, 16, [100, 3000]
    B, T = 2, 3000 + n
    k, v = synth.history(B, T, 33, 2)
    cache = gpu_cache(mg, kind, B, 2048, k, v, p0s)
    before = cache.k[1].clone(), cache.v[1].clone()
    blk_k = torch.stack([k[b, p:p + n] for b, p in enumerate(p0s)]).cuda().contiguous()
    blk_v = torch.stack([v[b, p:p + n] for b, p in enumerate(p0s)]).cuda().contiguous()
    err = mg.error_word()
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    mg.mg_kv_commit(mg.make_layer(kind), cache, torch.tensor(p0s, dtype=torch.int32, device="cuda"),
                    torch.tensor([3, n + 1], dtype=torch.int32, device="cuda"), blk_k, blk_v, err,
                    pos_next=nxt)
    torch.cuda.synchronize()
    check_err(err, DERR_COUNT)
    assert nxt.tolist() == [103, 3000]
    assert torch.equal(cache.k[1], before[0]) and torch.equal(cache.v[1], before[1])
    kc, vc = oracle_cache(kind, 2048, k[0], v[0], 103)
    assert np.array_equal(bits_of(cache.k[0]), kc)


@pytest.mark.parametrize("kind", [0, 1])
def test_speculative_rounds_against_linear_history(mg, kind):
    """Three rounds of verify + commit on two sequences with different
    acceptance; drafts past the accepted prefix are junk.  Every verify
    output is checked against the oracle over the linear history of kept
    tokens plus the block, the final cache bit for bit, and a decode after
    the last round against the oracle."""
    n, B = 16, 2
    p_start = [2030, 4090]        # the first rounds cross the ring wrap
    accept = [[4, 16, 1], [16, 0, 9]]  # tokens kept per round (0: anchor rejected too)
    T = max(p + sum(a) for p, a in zip(p_start, accept)) + n + 1
    slots = 2048 if kind == 0 else T
    li = 2 if kind == 0 else 3
    k, v = synth.history(B, T, 34, li)
    lay = mg.make_layer(kind)
    olay = orc.layer(oracle_kind(kind))
    cache = gpu_cache(mg, kind, B, slots, k, v, p_start)
    pos = torch.tensor(p_start, dtype=torch.int32, device="cuda")
    nxt = torch.empty_like(pos)
    err = mg.error_word()
    ws = mg.workspace(mg.OP_VERIFY, lay, B, n, T)
    p_host = list(p_start)
    for r in range(3):
        jk, jv = synth.history(B, n, 40 + r, li)
        q = synth.queries(B, n, 50 + r, li)
        counts = [accept[b][r] for b in range(B)]
        # the block: the true continuation up to the count, junk after it
        blk_k = torch.stack([torch.cat([k[b, p_host[b]:p_host[b] + counts[b]], jk[b, counts[b]:]])
                             for b in range(B)])
        blk_v = torch.stack([torch.cat([v[b, p_host[b]:p_host[b] + counts[b]], jv[b, counts[b]:]])
                             for b in range(B)])
        o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
        kb, vb = blk_k.cuda().contiguous(), blk_v.cuda().contiguous()
        mg.mg_attn_verify(lay, cache, pos, T, q.cuda().contiguous(), kb, vb, o, ws, err)
        mg.mg_kv_commit(lay, cache, pos, torch.tensor(counts, dtype=torch.int32, device="cuda"),
                        kb, vb, err, pos_next=nxt)
        pos.copy_(nxt)
        torch.cuda.synchronize()
        check_err(err)
        for b in range(B):
            p0 = p_host[b]
            hk = torch.cat([k[b, :p0], blk_k[b]])
            hv = torch.cat([v[b, :p0], blk_v[b]])
            ref = orc.attention(olay, hk, hv, list(range(p0, p0 + n)), q[b])
            compare(o[b], ref, f"kind {kind} round {r} b {b} p0 {p0}")
            p_host[b] += counts[b]
    assert pos.tolist() == p_host
    for b in range(B):
        kc, vc = oracle_cache(kind, slots, k[b], v[b], p_host[b])
        assert np.array_equal(bits_of(cache.k[b]), kc), f"K cache of sequence {b}"
        assert np.array_equal(bits_of(cache.v[b]), vc), f"V cache of sequence {b}"
    # one decode token after the last round, on the true continuation
    qd = synth.queries(B, 1, 60, li)[:, 0]
    mg.mg_kv_append(lay, cache, pos, torch.stack([k[b, p:p + 1] for b, p in enumerate(p_host)])
                    .cuda().contiguous(),
                    torch.stack([v[b, p:p + 1] for b, p in enumerate(p_host)]).cuda().contiguous(),
                    err)
    od = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    mg.mg_attn_decode(lay, cache, pos, T, qd.cuda().contiguous(), od,
                      mg.workspace(mg.OP_DECODE, lay, B, 1, T), err)
    torch.cuda.synchronize()
    check_err(err)
    for b, p in enumerate(p_host):
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], qd[b:b + 1])[0]
        compare(od[b], ref, f"kind {kind} decode after rounds b {b} p {p}")


def test_commit_layers_equals_per_layer_commits(mg):
    """One launch into four layers (local, local, local, global) gives the
    caches the oracle expects for each layer, the same as four commits."""
    kinds = [0, 0, 0, 1]
    p0s, counts, n = [2041, 5000], [9, 3], 16
    B, T = len(p0s), max(p0s) + n
    ks, vs, blocks_k, blocks_v, caches = [], [], [], [], []
    for l, kind in enumerate(kinds):
        k, v = synth.history(B, T, 70 + l, l)
        jk, jv = synth.history(B, n, 80 + l, l)
        bk = torch.stack([torch.cat([k[b, p:p + c], jk[b, c:]])
                          for b, (p, c) in enumerate(zip(p0s, counts))])
        bv = torch.stack([torch.cat([v[b, p:p + c], jv[b, c:]])
                          for b, (p, c) in enumerate(zip(p0s, counts))])
        ks.append(k)
        vs.append(v)
        blocks_k.append(bk)
        blocks_v.append(bv)
        caches.append(gpu_cache(mg, kind, B, 2048 if kind == 0 else T, k, v, p0s))
    err = mg.error_word()
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    mg.mg_kv_commit_layers([mg.make_layer(kd) for kd in kinds], caches,
                           torch.tensor(p0s, dtype=torch.int32, device="cuda"),
                           torch.tensor(counts, dtype=torch.int32, device="cuda"),
                           torch.stack(blocks_k).cuda().contiguous(),
                           torch.stack(blocks_v).cuda().contiguous(), err, pos_next=nxt)
    torch.cuda.synchronize()
    check_err(err)
    assert nxt.tolist() == [p + c for p, c in zip(p0s, counts)]
    for l, kind in enumerate(kinds):
        slots = 2048 if kind == 0 else T
        for b in range(B):
            kc, vc = oracle_cache(kind, slots, ks[l][b], vs[l][b], p0s[b])
            orc.cache_commit(oracle_kind(kind), kc, vc, p0s[b], counts[b], blocks_k[l][b],
                             blocks_v[l][b])
            assert np.array_equal(bits_of(caches[l].k[b]), kc), f"layer {l} K of sequence {b}"
            assert np.array_equal(bits_of(caches[l].v[b]), vc), f"layer {l} V of sequence {b}"
