"""The workloads at their full sizes, run the way bench.py runs them, checked
against the fp64 oracle on sampled outputs.

One local and one global layer of the 52-layer stack stand for their kinds:
every layer of a kind runs the same kernels with the same shapes, and the
seeds follow the layer index (layer 2 is local, layer 3 global).  Where the
oracle cannot recompute every output in seconds, whole (sequence, token)
rows are sampled: first and last rows, ring-wrap neighbourhoods and a
spread of the rest.
"""
import numpy as np
import pytest
import torch

from gpu_util import check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

LAYERS = [(0, 2), (1, 3)]  # (kind, layer index)


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def fill(mg, kind, k, v, T, capacity):
    """Cache after appending positions 0..T-1 of every sequence."""
    B = k.shape[0]
    cache = mg.KVCache(kind, B, capacity)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    lo = 0 if kind == 1 else max(0, T - 2048)
    mg.mg_kv_append(lay, cache, torch.tensor([lo] * B, dtype=torch.int32, device="cuda"),
                    k[:, lo:T].cuda().contiguous(), v[:, lo:T].cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err)
    return cache


@pytest.mark.parametrize("B", [1, 4, 16])
def test_decode_sweep_32k(mg, B):
    """Context 32768 pre-filled, 128 decode steps at p = 32768..32895 through
    mg_append_decode (as the benchmark's step does); every output of steps 0
    and 127 and of sequences 0 / B-1 at step 64 is checked."""
    T0, steps = 32768, 128
    cap = T0 + steps
    for kind, li in LAYERS:
        k, v = synth.history(B, cap, 1, li)
        q = synth.queries(B, steps, 1, li)
        cache = fill(mg, kind, k, v, T0, cap)
        lay = mg.make_layer(kind)
        ws = mg.workspace(mg.OP_DECODE, lay, B, 1, cap)
        err = mg.error_word()
        o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
        kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
        olay = orc.layer(oracle_kind(kind))
        for i in range(steps):
            p = T0 + i
            pos = torch.tensor([p] * B, dtype=torch.int32, device="cuda")
            mg.mg_append_decode(lay, cache, pos, cap, qd[:, i].contiguous(),
                                kd[:, p:p + 1].contiguous(), vd[:, p:p + 1].contiguous(), o, ws, err)
            if i in (0, 64, 127):
                torch.cuda.synchronize()
                check_err(err)
                bs = range(B) if i != 64 else sorted({0, B - 1})
                for b in bs:
                    ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], q[b, i:i + 1])[0]
                    compare(o[b], ref, f"kind {kind} B {B} b {b} step {i}")


@pytest.mark.parametrize("B", [1, 2, 8])
def test_verify_131k(mg, B):
    """16 draft tokens at p0 = 131072 against a 131072-token cache (the
    benchmark's verify leg); sequences 0 and B-1 checked in full."""
    T0, n = 131072, 16
    for kind, li in LAYERS:
        k, v = synth.history(B, T0 + n, 2, li)
        q = synth.queries(B, n, 2, li)
        cache = fill(mg, kind, k, v, T0, T0 + n)
        lay = mg.make_layer(kind)
        ws = mg.workspace(mg.OP_VERIFY, lay, B, n, T0 + n)
        err = mg.error_word()
        o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
        mg.mg_attn_verify(lay, cache, torch.tensor([T0] * B, dtype=torch.int32, device="cuda"),
                          T0 + n, q.cuda().contiguous(), k[:, T0:].cuda().contiguous(),
                          v[:, T0:].cuda().contiguous(), o, ws, err)
        torch.cuda.synchronize()
        check_err(err)
        olay = orc.layer(oracle_kind(kind))
        for b in sorted({0, B - 1}):
            ref = orc.attention(olay, k[b], v[b], list(range(T0, T0 + n)), q[b])
            compare(o[b], ref, f"kind {kind} B {B} b {b}")


def chunked_prefill(mg, kind, k, v, q, chunk, capacity, rows_per_chunk, seed):
    """Prefill the whole history in chunks (prefill, then append, per chunk)
    and return (sampled positions, their outputs)."""
    T = k.shape[1]
    cache = mg.KVCache(kind, 1, capacity)
    lay = mg.make_layer(kind)
    ws = mg.workspace(mg.OP_PREFILL, lay, 1, chunk, T)
    err = mg.error_word()
    o = torch.empty((1, chunk, 32, 128), dtype=torch.bfloat16, device="cuda")
    kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
    rng = np.random.default_rng(seed)
    picked, outs = [], []
    for c0 in range(0, T, chunk):
        pos = torch.tensor([c0], dtype=torch.int32, device="cuda")
        kn, vn = kd[:, c0:c0 + chunk].contiguous(), vd[:, c0:c0 + chunk].contiguous()
        mg.mg_attn_prefill(lay, cache, pos, c0 + chunk, qd[:, c0:c0 + chunk].contiguous(), kn, vn, o,
                           ws, err)
        rows = sorted({0, 1, 2047, 2048, chunk - 1} | set(rng.choice(chunk, rows_per_chunk, False)))
        rows = [r for r in rows if r < chunk]
        picked += [c0 + r for r in rows]
        outs.append(o[0, rows].clone())
        mg.mg_kv_append(lay, cache, pos, kn, vn, err)
    torch.cuda.synchronize()
    check_err(err)
    return cache, picked, torch.cat(outs)


def test_prefill_32k_chunks_4096(mg):
    """32768-token prompt in 4096-token chunks, one local and one global
    layer, batch 1; ~40 rows per chunk checked (all 32 heads)."""
    T, chunk = 32768, 4096
    for kind, li in LAYERS:
        k, v = synth.history(1, T, 3, li)
        q = synth.queries(1, T, 3, li)
        _, picked, outs = chunked_prefill(mg, kind, k, v, q, chunk, T, 35, seed=li)
        ref = orc.attention(orc.layer(oracle_kind(kind)), k[0], v[0], picked, q[0, picked])
        compare(outs, ref, f"prefill 32K kind {kind}")


def test_full_context_131k(mg):
    """131072-token prompt in 8192-token chunks, then 512 decode steps
    (positions 131072..131583), one local and one global layer, batch 1;
    sampled prefill rows and decode steps 0, 255, 511 checked."""
    T, chunk, steps = 131072, 8192, 512
    cap = T + steps
    for kind, li in LAYERS:
        k, v = synth.history(1, cap, 4, li)
        q = synth.queries(1, cap, 4, li)
        cache, picked, outs = chunked_prefill(mg, kind, k[:, :T], v[:, :T], q[:, :T], chunk, cap,
                                              3, seed=10 + li)
        olay = orc.layer(oracle_kind(kind))
        ref = orc.attention(olay, k[0, :T], v[0, :T], picked, q[0, picked])
        compare(outs, ref, f"full-context prefill kind {kind}")
        lay = mg.make_layer(kind)
        ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, cap)
        err = mg.error_word()
        o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
        kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
        for i in range(steps):
            p = T + i
            pos = torch.tensor([p], dtype=torch.int32, device="cuda")
            mg.mg_append_decode(lay, cache, pos, cap, qd[:, p].contiguous(), kd[:, p:p + 1].contiguous(),
                                vd[:, p:p + 1].contiguous(), o, ws, err)
            if i in (0, 255, 511):
                torch.cuda.synchronize()
                check_err(err)
                r = orc.attention(olay, k[0, :p + 1], v[0, :p + 1], [p], q[0, p:p + 1])[0]
                compare(o[0], r, f"full-context decode kind {kind} step {i}")
