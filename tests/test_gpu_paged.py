"""Paged global cache: sequences of different lengths share one pool of pages
through a page table ("Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse
Glimmer", "窄缓存为长上下文留出空间").  Pools are compared bit for bit with the
oracle's paged store, attention outputs against the oracle over each
sequence's linear history, and decode also bit for bit against the same call
on a linear cache."""
import numpy as np
import pytest
import torch

from gpu_util import bits_of, check_err, compare
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

GLOBAL = 1


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def shuffled_tables(B, lengths, capacity, ps, num_pages, seed):
    """Every sequence gets the pages its length needs, drawn from a random
    permutation of the pool; entries past a sequence's length stay -1."""
    rng = np.random.default_rng(seed)
    perm = list(rng.permutation(num_pages))
    table = np.full((B, capacity // ps), -1, np.int32)
    for b, n in enumerate(lengths):
        for j in range((n + ps - 1) // ps):
            table[b, j] = perm.pop()
    return table


def paged_cache(mg, B, lengths, capacity, ps, num_pages, k, v, seed=0):
    """A paged cache holding positions [0, lengths[b]) of each sequence,
    appended through the library, plus the oracle's pools for the same."""
    cache = mg.PagedKVCache(B, capacity, num_pages, ps)
    table = shuffled_tables(B, lengths, capacity, ps, num_pages, seed)
    cache.table.copy_(torch.from_numpy(table))
    lay = mg.make_layer(GLOBAL)
    err = mg.error_word()
    kp = np.zeros((num_pages, 2, ps, 128), np.uint16)
    vp = np.zeros_like(kp)
    # append each sequence in two uneven pieces (the second crossing a page)
    for b, n in enumerate(lengths):
        cut = min(n, 300)
        for a, z in ((0, cut), (cut, n)):
            if z <= a:
                continue
            pos = torch.full((B,), -1, dtype=torch.int32, device="cuda")
            pos[b] = a
            kn = torch.zeros((B, z - a, 2, 128), dtype=torch.bfloat16)
            vn = torch.zeros_like(kn)
            kn[b] = k[b, a:z]
            vn[b] = v[b, a:z]
            mg.mg_kv_append(lay, cache, pos, kn.cuda().contiguous(), vn.cuda().contiguous(), err)
            orc.paged_append(kp, vp, table[b], ps, a, k[b, a:z], v[b, a:z])
    torch.cuda.synchronize()
    # the other sequences were given pos -1: each such call flags a position
    # error and writes nothing for them, which is what the pools show
    assert int(err.item()) & ~mg.DERR_POSITION == 0, hex(int(err.item()))
    err.zero_()
    return cache, table, kp, vp


def test_paged_append_pools_bit_exact(mg):
    ps, B, cap, pool = 256, 3, 4096, 24
    lengths = [300, 1020, 5]
    k, v = synth.history(B, cap, 90, 3)
    cache, table, kp, vp = paged_cache(mg, B, lengths, cap, ps, pool, k, v)
    assert np.array_equal(bits_of(cache.k), kp)
    assert np.array_equal(bits_of(cache.v), vp)
    # a commit of 7 of 16 block tokens lands through the table too
    err = mg.error_word()
    p0 = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([7, 16, 0], dtype=torch.int32, device="cuda")
    blk_k = torch.stack([k[b, n:n + 16] for b, n in enumerate(lengths)])
    blk_v = torch.stack([v[b, n:n + 16] for b, n in enumerate(lengths)])
    # sequence 1's committed tokens 1020..1035 cross into logical page 4
    free = sorted(set(range(pool)) - set(table[table >= 0].tolist()))
    assert table[1, 4] == -1
    table[1, 4] = free[0]
    cache.table.copy_(torch.from_numpy(table))
    mg.mg_kv_commit(mg.make_layer(GLOBAL), cache, p0, cnt, blk_k.cuda().contiguous(),
                    blk_v.cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err)
    for b, n in enumerate(lengths):
        c = int(cnt[b])
        if c:
            orc.paged_append(kp, vp, table[b], ps, n, blk_k[b, :c], blk_v[b, :c])
    assert np.array_equal(bits_of(cache.k), kp)
    assert np.array_equal(bits_of(cache.v), vp)


@pytest.mark.parametrize("ps", [256, 512])
@pytest.mark.parametrize("fused", [False, True])
def test_paged_decode_against_oracle_and_linear(mg, ps, fused):
    B, cap = 3, 8192
    lengths = [700, 4097, 2050]           # the query's own token is at lengths[b]
    pool = sum((n + ps) // ps + 1 for n in lengths) + 3
    k, v = synth.history(B, cap, 91, 3)
    q = synth.queries(B, 1, 91, 3)[:, 0]
    hist = [n if fused else n + 1 for n in lengths]  # the query token's row first, unless fused
    cache, table, _, _ = paged_cache(mg, B, hist, cap, ps, pool, k, v, seed=ps)
    # the fused call writes the query token into the page of its position
    for b, n in enumerate(lengths):
        if table[b, n // ps] < 0:
            free = sorted(set(range(pool)) - set(table[table >= 0].tolist()))
            table[b, n // ps] = free[0]
    cache.table.copy_(torch.from_numpy(table))
    lay = mg.make_layer(GLOBAL)
    max_len = max(lengths) + 1
    pos = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    err = mg.error_word()
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, max_len)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.stack([k[b, n:n + 1] for b, n in enumerate(lengths)]).cuda().contiguous()
    vn = torch.stack([v[b, n:n + 1] for b, n in enumerate(lengths)]).cuda().contiguous()
    qd = q.cuda().contiguous()
    if fused:
        mg.mg_append_decode(lay, cache, pos, max_len, qd, kn, vn, o, ws, err)
    else:
        mg.mg_attn_decode(lay, cache, pos, max_len, qd, o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(orc.GLOBAL)
    for b, n in enumerate(lengths):
        ref = orc.attention(olay, k[b, :n + 1], v[b, :n + 1], [n], q[b:b + 1])[0]
        compare(o[b], ref, f"paged decode ps {ps} b {b} p {n}")
    # the same call on a linear cache gives the same bits (same splits, same tiles)
    lin = mg.KVCache(GLOBAL, B, cap)
    for b, n in enumerate(lengths):
        lin.k[b, :, :n + 1] = k[b, :n + 1].transpose(0, 1).cuda()
        lin.v[b, :, :n + 1] = v[b, :n + 1].transpose(0, 1).cuda()
    o2 = torch.empty_like(o)
    mg.mg_attn_decode(lay, lin, pos, max_len, qd, o2, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    assert torch.equal(o, o2)


@pytest.mark.parametrize("ps", [256, 512])
@pytest.mark.parametrize("op,p0s,n", [("verify", [1000, 3333], 16), ("verify", [256, 5000], 5),
                                      ("prefill", [1300, 40], 700), ("prefill", [512, 0], 300)])
def test_paged_verify_and_prefill_against_oracle(mg, ps, op, p0s, n):
    B, cap = len(p0s), 6144
    pool = sum((p + n + ps - 1) // ps for p in p0s) + 2
    k, v = synth.history(B, cap, 92, 3)
    q = synth.queries(B, n, 92, 3)
    # the cache holds positions < p0[b]; the block is passed in
    cache, table, _, _ = paged_cache(mg, B, p0s, cap, ps, pool, k, v, seed=7 * ps + n)
    lay = mg.make_layer(GLOBAL)
    max_len = max(p0s) + n
    op_id = mg.OP_VERIFY if op == "verify" else mg.OP_PREFILL
    ws = mg.workspace(op_id, lay, B, n, max_len)
    o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    kn = torch.stack([k[b, p:p + n] for b, p in enumerate(p0s)]).cuda().contiguous()
    vn = torch.stack([v[b, p:p + n] for b, p in enumerate(p0s)]).cuda().contiguous()
    pos = torch.tensor(p0s, dtype=torch.int32, device="cuda")
    fn = mg.mg_attn_verify if op == "verify" else mg.mg_attn_prefill
    fn(lay, cache, pos, max_len, q.cuda().contiguous(), kn, vn, o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(orc.GLOBAL)
    for b, p0 in enumerate(p0s):
        ref = orc.attention(olay, k[b, :p0 + n], v[b, :p0 + n], list(range(p0, p0 + n)), q[b])
        compare(o[b], ref, f"paged {op} ps {ps} b {b} p0 {p0} n {n}")


def test_page_entry_outside_pool_is_flagged(mg):
    # A table entry past the pool is caught by the kernels (page 0 is read
    # instead, no access leaves the pool): the error word says so.
    ps, B, cap, pool = 256, 1, 2048, 8
    k, v = synth.history(B, cap, 93, 3)
    cache, table, _, _ = paged_cache(mg, B, [1000], cap, ps, pool, k, v)
    table[0, 1] = pool + 3
    cache.table.copy_(torch.from_numpy(table))
    lay = mg.make_layer(GLOBAL)
    err = mg.error_word()
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([999], dtype=torch.int32, device="cuda")
    mg.mg_attn_decode(lay, cache, pos, 1000, synth.queries(B, 1, 93, 3)[:, 0].cuda().contiguous(), o,
                      mg.workspace(mg.OP_DECODE, lay, B, 1, 1000), err)
    torch.cuda.synchronize()
    assert int(err.item()) & mg.DERR_PAGE
    assert torch.isfinite(o.float()).all()
