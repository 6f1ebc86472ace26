"""Decode attention on the GPU against the fp64 oracle: ragged positions
around tile and ring boundaries, mixed batches, the 256-step two-layer
decode across the ring wrap with the cache checked bit for bit after every
step, and sampled checks at 32K and 128K context."""
import numpy as np
import pytest
import torch

from gpu_util import bits_of, cache_expected, check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def fill_for_decode(mg, kind, k, v, positions, capacity):
    """Cache whose state is what appending positions 0..p_b gives (for the
    ring: the last 2048 of them).  Returns the cache."""
    B = k.shape[0]
    cache = mg.KVCache(kind, B, capacity)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    if kind == 1:
        n = k.shape[1]
        pos0 = [0] * B
    else:
        n = 2048
        pos0 = [max(0, p - 2047) for p in positions]
    kn = torch.stack([k[b, p:p + n] for b, p in enumerate(pos0)]).cuda().contiguous()
    vn = torch.stack([v[b, p:p + n] for b, p in enumerate(pos0)]).cuda().contiguous()
    mg.mg_kv_append(lay, cache, torch.tensor(pos0, dtype=torch.int32, device="cuda"), kn, vn, err)
    torch.cuda.synchronize()
    check_err(err)
    return cache


def decode_once(mg, kind, cache, positions, q, max_len):
    lay = mg.make_layer(kind)
    B = q.shape[0]
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, max_len)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    mg.mg_attn_decode(lay, cache, torch.tensor(positions, dtype=torch.int32, device="cuda"), max_len,
                      q.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    return o, err


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("positions", [[0, 1, 63], [64, 65, 127], [2046, 2047, 2048],
                                       [3000, 4095, 4100], [129, 2500, 63]])
def test_decode_ragged_positions(mg, kind, positions):
    B = len(positions)
    T = max(max(0, p - 2047) for p in positions) + 2048 if kind == 0 else max(positions) + 1
    k, v = synth.history(B, T, 7, 2 if kind == 0 else 3)
    q = synth.queries(B, 1, 7, 2 if kind == 0 else 3)[:, 0]
    cache = fill_for_decode(mg, kind, k, v, positions, capacity=T)
    max_len = max(positions) + 1
    o, err = decode_once(mg, kind, cache, positions, q, max_len)
    check_err(err)
    lay = orc.layer(oracle_kind(kind))
    for b, p in enumerate(positions):
        ref = orc.attention(lay, k[b, :p + 1], v[b, :p + 1], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"kind {kind} b {b} p {p}")


def test_decode_position_beyond_max_len_is_flagged(mg):
    k, v = synth.history(2, 300, 8, 3)
    q = synth.queries(2, 1, 8, 3)[:, 0]
    cache = fill_for_decode(mg, 1, k, v, [100, 299], capacity=300)
    o, err = decode_once(mg, 1, cache, [100, 299], q, max_len=200)  # 299 >= max_len
    check_err(err, mg.DERR_POSITION)
    ref = orc.attention(orc.layer(orc.GLOBAL), k[0, :101], v[0, :101], [100], q[:1])[0]
    compare(o[0], ref, "valid sequence next to a rejected one")
    assert float(o[1].float().abs().max()) == 0.0


@pytest.mark.parametrize("fused", [False, True])
def test_pr1_two_layer_decode_across_ring_wrap(mg, fused):
    """One local (window 2048, RoPE 1e4) and one global layer, batch 1, seed 0:
    cache pre-filled for positions 0..1999, then 256 single-token steps at
    p = 2000..2255 (append, then decode -- as two calls, or fused in
    mg_append_decode), every output compared with the oracle and both caches
    compared bit for bit after every step."""
    seed, P0, steps = 0, 2000, 256
    T = P0 + steps
    layers = [(0, 0), (1, 3)]  # (kind, layer index for the seed)
    state = []
    for kind, li in layers:
        k, v = synth.history(1, T, seed, li)
        q = synth.queries(1, steps, seed, li)
        cache = mg.KVCache(kind, 1, T)
        lay = mg.make_layer(kind)
        err = mg.error_word()
        mg.mg_kv_append(lay, cache, torch.tensor([0], dtype=torch.int32, device="cuda"),
                        k[:, :P0].cuda().contiguous(), v[:, :P0].cuda().contiguous(), err)
        ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, T)
        exp_k = np.zeros((2, cache.slots, 128), np.uint16)
        exp_v = np.zeros_like(exp_k)
        orc.cache_append(oracle_kind(kind), exp_k, exp_v, 0, k[0, :P0], v[0, :P0])
        state.append(dict(kind=kind, k=k, v=v, q=q, cache=cache, lay=lay, err=err, ws=ws,
                          kd=k.cuda(), vd=v.cuda(), qd=q.cuda(), exp_k=exp_k, exp_v=exp_v,
                          olay=orc.layer(oracle_kind(kind))))
    o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    worst = 0.0
    for i in range(steps):
        p = P0 + i
        pos = torch.tensor([p], dtype=torch.int32, device="cuda")
        for s in state:
            kn, vn = s["kd"][:, p:p + 1].contiguous(), s["vd"][:, p:p + 1].contiguous()
            if fused:
                mg.mg_append_decode(s["lay"], s["cache"], pos, T, s["qd"][:, i].contiguous(), kn, vn,
                                    o, s["ws"], s["err"])
            else:
                mg.mg_kv_append(s["lay"], s["cache"], pos, kn, vn, s["err"])
                mg.mg_attn_decode(s["lay"], s["cache"], pos, T, s["qd"][:, i].contiguous(), o,
                                  s["ws"], s["err"])
            orc.cache_append(oracle_kind(s["kind"]), s["exp_k"], s["exp_v"], p, s["k"][0, p:p + 1],
                             s["v"][0, p:p + 1])
            ref = orc.attention(s["olay"], s["k"][0, :p + 1], s["v"][0, :p + 1], [p], s["q"][:, i])[0]
            err_abs, _, _ = compare(o[0], ref, f"kind {s['kind']} step {i} p {p}")
            worst = max(worst, err_abs)
            assert np.array_equal(bits_of(s["cache"].k[0]), s["exp_k"]), f"K cache step {i}"
            assert np.array_equal(bits_of(s["cache"].v[0]), s["exp_v"]), f"V cache step {i}"
    for s in state:
        check_err(s["err"])


@pytest.mark.parametrize("kind", [0, 1])
def test_append_decode_mixed_batch(mg, kind):
    """Fused append + decode for a batch whose sequences sit at different
    positions (some below the window, one right at the ring wrap)."""
    positions = [5, 2047, 2048, 3001]
    B = len(positions)
    T = max(positions) + 1
    k, v = synth.history(B, T, 9, 2 if kind == 0 else 3)
    q = synth.queries(B, 1, 9, 2 if kind == 0 else 3)[:, 0]
    # cache holding positions < p_b (ring: the last 2048 of them)
    cache = mg.KVCache(kind, B, T)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    for b, p in enumerate(positions):
        lo = max(0, p - 2048) if kind == 0 else 0
        one = mg.KVCache(kind, 1, T)
        mg.mg_kv_append(lay, one, torch.tensor([lo], dtype=torch.int32, device="cuda"),
                        k[b:b + 1, lo:p].cuda().contiguous(), v[b:b + 1, lo:p].cuda().contiguous(), err)
        cache.k[b].copy_(one.k[0])
        cache.v[b].copy_(one.v[0])
    kn = torch.stack([k[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
    vn = torch.stack([v[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, T)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    mg.mg_append_decode(lay, cache, torch.tensor(positions, dtype=torch.int32, device="cuda"), T,
                        q.cuda().contiguous(), kn, vn, o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(oracle_kind(kind))
    for b, p in enumerate(positions):
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"kind {kind} b {b} p {p}")
        lo = max(0, p - 2047) if kind == 0 else 0
        kc, vc = cache_expected(kind, cache.slots, k[b], v[b], [(lo, p + 1 - lo)])
        # slots never written stay zero on both sides
        assert np.array_equal(bits_of(cache.k[b]), kc), f"K cache b {b}"
        assert np.array_equal(bits_of(cache.v[b]), vc), f"V cache b {b}"


@pytest.mark.parametrize("B,T", [(1, 131072 + 64), (3, 5000), (40, 700), (160, 900)])
def test_global_decode_repeats_exactly(mg, B, T):
    """Global decode at batch 1, 3, 40 and 160 (148, 49, 3 and 1 splits per
    KV head; a single split writes the output without partials or combine):
    eager calls and graph replays give the same bits, sampled rows match the
    oracle, and the kernel count the library reports fits the split count."""
    lay = mg.make_layer(1)
    positions = [T - 1 - (37 * b) % (T // 2) for b in range(B)]
    k, v = synth.history(B, T, 9, 3)
    q = synth.queries(B, 1, 9, 3)[:, 0]
    cache = fill_for_decode(mg, 1, k, v, positions, capacity=T)
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, T)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    qd = q.cuda().contiguous()
    outs = []
    for _ in range(2):
        mg.mg_attn_decode(lay, cache, pos, T, qd, o, ws, err)
        torch.cuda.synchronize()
        outs.append(o.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mg.mg_attn_decode(lay, cache, pos, T, qd, o, ws, err)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check_err(err)
    outs.append(o.clone())
    assert all(torch.equal(outs[0], x) for x in outs[1:])
    assert mg.mg_decode_kernel_count(lay, B, T) == (1 if B == 160 else 2)
    olay = orc.layer(orc.GLOBAL)
    for b in sorted({0, B // 2, B - 1}):
        p = positions[b]
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"B {B} b {b} p {p}")


@pytest.mark.parametrize("B", [4, 9, 16])
@pytest.mark.parametrize("fused", [False, True])
def test_local_decode_larger_batches(mg, B, fused):
    """Local decode with more (sequence, KV head) pairs than one wave of
    16-CTA clusters holds: clusters of 8 or 4 CTAs walking their ring piece
    in rounds of 128 slots (online softmax across rounds).  Ragged
    positions leave some CTAs and rounds without keys and some rounds partly
    filled; fused=True also appends the token's own row."""
    positions = [0, 1, 100, 127, 128, 255, 256, 511, 513, 1023, 1024, 2047, 2048, 3000, 4095,
                 5000][:B]
    T = max(positions) + 1
    k, v = synth.history(B, T, 13, 2)
    q = synth.queries(B, 1, 13, 2)[:, 0]
    lay = mg.make_layer(0)
    cache = mg.KVCache(0, B, T)
    err = mg.error_word()
    # the ring of each sequence: positions up to p - 1 (fused) or p
    for b, p in enumerate(positions):
        top = p if fused else p + 1
        lo = max(0, top - 2048)
        if top > lo:
            one = mg.KVCache(0, 1, T)
            mg.mg_kv_append(lay, one, torch.tensor([lo], dtype=torch.int32, device="cuda"),
                            k[b:b + 1, lo:top].cuda().contiguous(), v[b:b + 1, lo:top].cuda().contiguous(),
                            err)
            cache.k[b].copy_(one.k[0])
            cache.v[b].copy_(one.v[0])
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, T)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    if fused:
        kn = torch.stack([k[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
        vn = torch.stack([v[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
        mg.mg_append_decode(lay, cache, pos, T, q.cuda().contiguous(), kn, vn, o, ws, err)
    else:
        mg.mg_attn_decode(lay, cache, pos, T, q.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(orc.LOCAL)
    for b, p in enumerate(positions):
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"B {B} b {b} p {p}")
    if fused:  # the ring holds each token's own row now
        for b, p in enumerate(positions):
            assert torch.equal(cache.k[b, :, p % 2048], k[b, p].cuda())
            assert torch.equal(cache.v[b, :, p % 2048], v[b, p].cuda())


@pytest.mark.parametrize("B,case", [(8, "x40"), (16, "sink")])
def test_local_decode_rounds_peaked(mg, B, case):
    """Peaked rows through the multi-round form: queries x40 (the running
    max moves between rounds), or a sink key in the last round of a CTA's
    piece (slots 1920..2047 in the 4-CTA clusters' last piece)."""
    p = 5000
    k, v = synth.history(B, p + 1, 14, 2)
    q = synth.queries(B, 1, 14, 2)[:, 0]
    if case == "x40":
        q = synth.scaled(q, 40.0)
    else:
        sink = p - ((p - 1990) % 2048)  # the position held in ring slot 1990
        k = synth.plant_sinks(k, [sink])
        q = synth.sink_queries(q)
    lay = mg.make_layer(0)
    cache = mg.KVCache(0, B, p + 1)
    err = mg.error_word()
    mg.mg_kv_append(lay, cache, torch.tensor([p - 2047] * B, dtype=torch.int32, device="cuda"),
                    k[:, p - 2047:].cuda().contiguous(), v[:, p - 2047:].cuda().contiguous(), err)
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, p + 1)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    mg.mg_attn_decode(lay, cache, torch.tensor([p] * B, dtype=torch.int32, device="cuda"), p + 1,
                      q.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    olay = orc.layer(orc.LOCAL)
    for b in range(B):
        ref = orc.attention(olay, k[b], v[b], [p], q[b:b + 1])[0]
        compare(o[b], ref, f"{case} B {B} b {b}")


@pytest.mark.parametrize("bases", [[2040], [100], [2040, 3000, 4090], [2040, 3000, 4090, 100]])
def test_append_decode_early_matches_plain(mg, bases):
    """mg_append_decode_ex with MG_EARLY_START: a local and a global layer
    decoded in turn for 24 steps (each call's previous kernel is the other
    layer's, which writes neither this cache nor the positions), captured in
    one CUDA graph so that the calls overlap as in a decode step.  Outputs
    and caches equal the plain mg_append_decode run bit for bit, and every
    step's outputs match the oracle."""
    B = len(bases)
    S = 24
    T = max(bases) + S
    layers = []
    for kind, li in ((0, 4), (1, 5)):
        k, v = synth.history(B, T, 21, li)
        q = synth.queries(B, S, 21, li)
        layers.append(dict(kind=kind, k=k, v=v, q=q, kd=k.cuda(), vd=v.cuda(), qd=q.cuda(),
                           lay=mg.make_layer(kind), ws=mg.workspace(mg.OP_DECODE, mg.make_layer(kind), B, 1, T),
                           fill=fill_for_decode(mg, kind, k[:, :max(bases)], v[:, :max(bases)],
                                                [p - 1 for p in bases], T)))
    pos_all = torch.tensor([[p + i for p in bases] for i in range(S)], dtype=torch.int32, device="cuda")
    kn_all = [torch.stack([torch.stack([L["kd"][b, p + i] for b, p in enumerate(bases)])[:, None]
                           for i in range(S)]).contiguous() for L in layers]
    vn_all = [torch.stack([torch.stack([L["vd"][b, p + i] for b, p in enumerate(bases)])[:, None]
                           for i in range(S)]).contiguous() for L in layers]
    q_all = [L["qd"].transpose(0, 1).contiguous() for L in layers]  # [S][B][32][128]

    def run(early):
        caches = []
        for L in layers:
            c = mg.KVCache(L["kind"], B, T)
            c.k.copy_(L["fill"].k)
            c.v.copy_(L["fill"].v)
            caches.append(c)
        outs = torch.zeros((S, 2, B, 32, 128), dtype=torch.bfloat16, device="cuda")
        err = mg.error_word()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(S):
                for li, L in enumerate(layers):
                    args = (L["lay"], caches[li], pos_all[i], T, q_all[li][i], kn_all[li][i], vn_all[li][i],
                            outs[i, li], L["ws"], err)
                    if early:
                        mg.mg_append_decode_ex(*args, mg.EARLY_START)
                    else:
                        mg.mg_append_decode(*args)
        g.replay()
        torch.cuda.synchronize()
        check_err(err)
        return outs, caches

    oa, ca = run(False)
    ob, cb = run(True)
    assert torch.equal(oa, ob), "early decode differs from the plain call"
    for x, y in zip(ca, cb):
        assert torch.equal(x.k, y.k) and torch.equal(x.v, y.v), "caches differ"
    for li, L in enumerate(layers):
        olay = orc.layer(oracle_kind(L["kind"]))
        for i in (0, S // 2, S - 1):
            for b, p in enumerate(bases):
                ref = orc.attention(olay, L["k"][b, :p + i + 1], L["v"][b, :p + i + 1], [p + i],
                                    L["q"][b, i:i + 1])[0]
                compare(ob[i, li, b], ref, f"layer kind {L['kind']} step {i} seq {b}")


@pytest.mark.parametrize("bases", [[2040], [100], [2040, 3000, 4090]])
def test_append_decode_overlap_chain_matches_plain(mg, bases):
    """MG_EARLY_START | MG_OVERLAP_NEXT on every call of a step of three local
    layers and one global layer, as a model's decode step orders them, for
    12 steps in one CUDA graph; a torch kernel between steps (the position
    update of a real loop) ends each chain, since a layer's next step reads
    the row this step appends.  Inside a step each call's loads run under
    the calls before it (at batch 1; larger batches ignore the flags for the
    local layers).  Outputs and caches equal the plain mg_append_decode run
    bit for bit, and sampled steps match the oracle."""
    B = len(bases)
    S = 12
    T = max(bases) + S
    kinds = (0, 0, 0, 1)
    layers = []
    for li, kind in enumerate(kinds):
        k, v = synth.history(B, T, 31, 10 + li)
        q = synth.queries(B, S, 31, 10 + li)
        layers.append(dict(kind=kind, k=k, v=v, q=q, kd=k.cuda(), qd=q.cuda(), vd=v.cuda(),
                           lay=mg.make_layer(kind), ws=mg.workspace(mg.OP_DECODE, mg.make_layer(kind), B, 1, T),
                           fill=fill_for_decode(mg, kind, k[:, :max(bases)], v[:, :max(bases)],
                                                [p - 1 for p in bases], T)))
    pos_all = torch.tensor([[p + i for p in bases] for i in range(S)], dtype=torch.int32, device="cuda")
    kn_all = [torch.stack([torch.stack([L["kd"][b, p + i] for b, p in enumerate(bases)])[:, None]
                           for i in range(S)]).contiguous() for L in layers]
    vn_all = [torch.stack([torch.stack([L["vd"][b, p + i] for b, p in enumerate(bases)])[:, None]
                           for i in range(S)]).contiguous() for L in layers]
    q_all = [L["qd"].transpose(0, 1).contiguous() for L in layers]  # [S][B][32][128]

    def run(flags):
        caches = []
        for L in layers:
            c = mg.KVCache(L["kind"], B, T)
            c.k.copy_(L["fill"].k)
            c.v.copy_(L["fill"].v)
            caches.append(c)
        outs = torch.zeros((S, len(layers), B, 32, 128), dtype=torch.bfloat16, device="cuda")
        steps_done = torch.zeros(1, dtype=torch.int32, device="cuda")
        err = mg.error_word()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(S):
                for li, L in enumerate(layers):
                    args = (L["lay"], caches[li], pos_all[i], T, q_all[li][i], kn_all[li][i], vn_all[li][i],
                            outs[i, li], L["ws"], err)
                    if flags:
                        mg.mg_append_decode_ex(*args, flags)
                    else:
                        mg.mg_append_decode(*args)
                steps_done.add_(1)  # a kernel without the flags between steps
        g.replay()
        torch.cuda.synchronize()
        check_err(err)
        assert int(steps_done.item()) == S
        return outs, caches

    oa, ca = run(0)
    ob, cb = run(mg.EARLY_START | mg.OVERLAP_NEXT)
    assert torch.equal(oa, ob), "overlapped decode differs from the plain calls"
    for x, y in zip(ca, cb):
        assert torch.equal(x.k, y.k) and torch.equal(x.v, y.v), "caches differ"
    for li, L in enumerate(layers):
        olay = orc.layer(oracle_kind(L["kind"]))
        for i in (0, S - 1):
            for b, p in enumerate(bases):
                ref = orc.attention(olay, L["k"][b, :p + i + 1], L["v"][b, :p + i + 1], [p + i],
                                    L["q"][b, i:i + 1])[0]
                compare(ob[i, li, b], ref, f"layer {li} kind {L['kind']} step {i} seq {b}")


def test_append_decode_early_broken_promise_stays_in_bounds(mg):
    """MG_EARLY_START right after a kernel that does write the cache (the
    promise broken on purpose, both layer kinds, batch 1):
    the result may use stale rows, but every access stays inside the cache,
    no error is flagged and the outputs are finite."""
    T = 3000
    for kind in (0, 1):
        k, v = synth.history(1, T + 2, 23, 6 + kind)
        q = synth.queries(1, 1, 23, 6 + kind)[:, 0]
        cache = fill_for_decode(mg, kind, k[:, :T], v[:, :T], [T - 1], T + 2)
        lay = mg.make_layer(kind)
        ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, T + 2)
        err = mg.error_word()
        pos = torch.tensor([T], dtype=torch.int32, device="cuda")
        kn = k[:, T:T + 1].contiguous().cuda()
        vn = v[:, T:T + 1].contiguous().cuda()
        qd = q.contiguous().cuda()
        o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            # the kernel just before the early-start call writes the cache row
            # at T, which the early start may read before that write lands
            mg.mg_kv_append(lay, cache, pos, kn, vn, err)
            mg.mg_append_decode_ex(lay, cache, pos, T + 2, qd, kn, vn, o, ws, err, mg.EARLY_START)
        g.replay()
        torch.cuda.synchronize()
        check_err(err)
        assert torch.isfinite(o.float()).all()
