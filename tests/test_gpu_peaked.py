"""Parity at large and small score magnitudes, where the online softmax and
the log-sum-exp merges take their rare branches.

Every case compares the CUDA path element by element with the fp64 oracle:
  * queries scaled by 1e-3 (flat rows: outputs near the mean of V), 1 and 40
    (scaled scores of standard deviation ~40: each new key tile can raise a
    row's running maximum by many units, so the tensor-core kernel rescales
    its output accumulator in TMEM, and the decode kernels' maxima jump);
  * a sink key scoring ~45 above every other key, placed in the key tile a
    row visits last (the tensor-core kernel walks cache tiles from the block
    start downwards, then the block's own tiles upwards; the decode kernels
    walk tiles upwards), or in one split / one ring piece only, so that the
    split partials and the cluster's per-piece partials differ in their
    log-sum-exp by tens of units and the merge weights underflow for all
    but one of them.
Sources: "深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？" §01 and
§04 (window, heads, the 16-token verify block); "Tomas Koutsky 解释了 Meta 如何
在 24 GB 的容量内容纳 Muse Glimmer", "长上下文仍然带来计算开销" (full attention in
global layers, chunked prompt processing).
"""
import pytest
import torch

from gpu_util import check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

FACTORS = [1e-3, 1.0, 40.0]


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def append_history(mg, kind, cache, k, v, lo, hi):
    """Append positions [lo[b], hi) of every sequence's history (one call)."""
    B = k.shape[0]
    n = hi - min(lo)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    assert all(hi - x == n for x in lo)
    kn = torch.stack([k[b, lo[b]:hi] for b in range(B)]).cuda().contiguous()
    vn = torch.stack([v[b, lo[b]:hi] for b in range(B)]).cuda().contiguous()
    mg.mg_kv_append(lay, cache, torch.tensor(lo, dtype=torch.int32, device="cuda"), kn, vn, err)
    torch.cuda.synchronize()
    check_err(err)


def decode_case(mg, kind, k, v, q, p):
    """Single-token decode at position p of every sequence (cache filled with
    positions <= p) against the oracle."""
    B = k.shape[0]
    cache = mg.KVCache(kind, B, p + 1)
    lo = max(0, p - 2047) if kind == 0 else 0
    append_history(mg, kind, cache, k, v, [lo] * B, p + 1)
    lay = mg.make_layer(kind)
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, p + 1)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    mg.mg_attn_decode(lay, cache, torch.tensor([p] * B, dtype=torch.int32, device="cuda"), p + 1,
                      q.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(oracle_kind(kind))
    for b in range(B):
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"decode kind {kind} b {b} p {p}")


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("factor", FACTORS)
def test_decode_scaled_queries(mg, kind, factor):
    # global: batch 1 at 40000 keys runs 148 splits and the wide combine
    B, p = (1, 39999) if kind == 1 else (2, 5000)
    li = 2 if kind == 0 else 3
    k, v = synth.history(B, p + 1, 41, li)
    q = synth.scaled(synth.queries(B, 1, 41, li)[:, 0], factor)
    decode_case(mg, kind, k, v, q, p)


@pytest.mark.parametrize("kind,p,sink", [
    (1, 39999, 5),       # first tile of split 0: one split's lse ~40 above the rest
    (1, 39999, 39996),   # the last tile its split visits: the running max jumps at the end
    (1, 2047, 2047),     # the query's own key, one split per KV head at batch 3
    (0, 5000, 3100),     # one ring piece of the cluster dominates the merge
    (0, 5000, 4998),     # the piece just below the query's slot
    (0, 1500, 0),        # ring not yet full
])
def test_decode_sink_key(mg, kind, p, sink):
    B = 3 if p == 2047 else 1
    li = 2 if kind == 0 else 3
    k, v = synth.history(B, p + 1, 42, li)
    k = synth.plant_sinks(k, [sink])
    q = synth.sink_queries(synth.queries(B, 1, 42, li)[:, 0])
    decode_case(mg, kind, k, v, q, p)


def verify_case(mg, kind, k, v, q, p0s, n):
    B = len(p0s)
    T = max(p0s) + n
    cache = mg.KVCache(kind, B, T)
    for b, p0 in enumerate(p0s):  # the ring / linear cache of positions < p0
        lo = max(0, p0 - 2048) if kind == 0 else 0
        one = mg.KVCache(kind, 1, T)
        append_history(mg, kind, one, k[b:b + 1], v[b:b + 1], [lo], p0)
        cache.k[b].copy_(one.k[0])
        cache.v[b].copy_(one.v[0])
    lay = mg.make_layer(kind)
    kn = torch.stack([k[b, p:p + n] for b, p in enumerate(p0s)])
    vn = torch.stack([v[b, p:p + n] for b, p in enumerate(p0s)])
    ws = mg.workspace(mg.OP_VERIFY, lay, B, n, T)
    o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    mg.mg_attn_verify(lay, cache, torch.tensor(p0s, dtype=torch.int32, device="cuda"), T,
                      q.cuda().contiguous(), kn.cuda().contiguous(), vn.cuda().contiguous(), o, ws,
                      err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(oracle_kind(kind))
    for b, p0 in enumerate(p0s):
        ref = orc.attention(olay, k[b, :p0 + n], v[b, :p0 + n], list(range(p0, p0 + n)), q[b])
        compare(o[b], ref, f"verify kind {kind} b {b} p0 {p0}")


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("factor", FACTORS)
def test_verify_scaled_queries(mg, kind, factor):
    p0s, n = [5000, 2100], 16
    li = 2 if kind == 0 else 3
    k, v = synth.history(2, max(p0s) + n, 43, li)
    q = synth.scaled(synth.queries(2, n, 43, li), factor)
    verify_case(mg, kind, k, v, q, p0s, n)


@pytest.mark.parametrize("kind,sinks", [
    (1, [5]),              # the lowest cache tile (its split's only one): split lse far apart
    (1, [4000, 5010]),     # a cache sink, then one inside the block for tokens >= 10
    (0, [3600]),           # one ring piece dominates the cluster merge
    (0, [4990, 5007]),     # ring sink, then a block sink (token 7 onwards)
])
def test_verify_sink_key(mg, kind, sinks):
    p0s, n = [5000], 16
    li = 2 if kind == 0 else 3
    k, v = synth.history(1, 5016, 44, li)
    vals = [synth.SINK_K * (1.0 + 0.5 * i) for i in range(len(sinks))]  # later sinks win
    k = synth.plant_sinks(k, sinks, values=vals)
    q = synth.sink_queries(synth.queries(1, n, 44, li))
    verify_case(mg, kind, k, v, q, p0s, n)


def prefill_case(mg, kind, k, v, q, chunk):
    """Prefill the whole history in chunks (append after each) and compare
    sampled rows of every chunk with the oracle."""
    B, T = k.shape[0], k.shape[1]
    cache = mg.KVCache(kind, B, T)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
    olay = orc.layer(oracle_kind(kind))
    for c0 in range(0, T, chunk):
        n = min(chunk, T - c0)
        kn, vn = kd[:, c0:c0 + n].contiguous(), vd[:, c0:c0 + n].contiguous()
        ws = mg.workspace(mg.OP_PREFILL, lay, B, n, c0 + n)
        o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
        e = mg.error_word()
        mg.mg_attn_prefill(lay, cache, torch.tensor([c0] * B, dtype=torch.int32, device="cuda"),
                           c0 + n, qd[:, c0:c0 + n].contiguous(), kn, vn, o, ws, e)
        mg.mg_kv_append(lay, cache, torch.tensor([c0] * B, dtype=torch.int32, device="cuda"), kn, vn,
                        err)
        torch.cuda.synchronize()
        check_err(e)
        rows = sorted(set(list(range(0, 24)) + list(range(n - 24, n)) + list(range(0, n, 29))))
        pos = [c0 + r for r in rows]
        ref = orc.attention(olay, k[0, :c0 + n], v[0, :c0 + n], pos, q[0, pos])
        compare(o[0, rows], ref, f"prefill kind {kind} chunk at {c0}")
    check_err(err)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("factor", FACTORS)
def test_prefill_scaled_queries(mg, kind, factor):
    T, chunk = (4500, 1500) if kind == 0 else (2600, 1000)
    li = 2 if kind == 0 else 3
    k, v = synth.history(1, T, 45, li)
    q = synth.scaled(synth.queries(1, T, 45, li), factor)
    prefill_case(mg, kind, k, v, q, chunk)


@pytest.mark.parametrize("kind,T,chunk,sinks", [
    # global: position 5 is in the last cache tile every later row visits;
    # 1800 lies in the block tile 768..1023 of the chunk at 1000, which rows
    # 1800..1999 visit last
    (1, 2600, 1000, [5, 1800]),
    # local: 2000 is in the window of rows up to 4047 and visited among the
    # last cache tiles of the chunk at 3000; 3300 is a block sink
    (0, 4500, 1500, [2000, 3300]),
])
def test_prefill_sink_keys(mg, kind, T, chunk, sinks):
    li = 2 if kind == 0 else 3
    k, v = synth.history(1, T, 46, li)
    k = synth.plant_sinks(k, sinks, values=[synth.SINK_K, 1.5 * synth.SINK_K])
    q = synth.sink_queries(synth.queries(1, T, 46, li))
    prefill_case(mg, kind, k, v, q, chunk)


@pytest.mark.parametrize("case", ["x40", "sink"])
def test_local_verify_rounds_peaked(mg, case):
    """A local verify batch large enough for the 4-CTA clusters whose CTAs
    walk their ring piece in rounds (8 sequences x 2 KV heads x 2 token
    groups), with queries x40 or a sink key held in a CTA's last round
    (ring slot 1990)."""
    B, n = 8, 16
    p0s = [5000 + 37 * b for b in range(B)]
    k, v = synth.history(B, max(p0s) + n, 47, 2)
    q = synth.queries(B, n, 47, 2)
    if case == "x40":
        q = synth.scaled(q, 40.0)
    else:
        for b, p0 in enumerate(p0s):  # the position each sequence's ring holds in slot 1990
            k = synth.plant_sinks(k, [(p0 - 1) - ((p0 - 1 - 1990) % 2048)], seq=b)
        q = synth.sink_queries(q)
    verify_case(mg, 0, k, v, q, p0s, n)
