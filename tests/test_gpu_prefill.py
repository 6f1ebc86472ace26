"""Causal chunked prefill on the tensor-core path against the oracle:
ragged chunk lengths, chunks after a filled cache (ring wrapped for local
layers), and chunked == unchunked."""
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


def run_prefill(mg, kind, cache, c0s, q, kn, vn, max_len):
    lay = mg.make_layer(kind)
    B, n = q.shape[0], q.shape[1]
    ws = mg.workspace(mg.OP_PREFILL, lay, B, n, max_len)
    o = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    mg.mg_attn_prefill(lay, cache, torch.tensor(c0s, dtype=torch.int32, device="cuda"), max_len,
                       q.cuda().contiguous(), kn.cuda().contiguous(), vn.cuda().contiguous(), o, ws,
                       err)
    torch.cuda.synchronize()
    return o, err


def prefill_chunks(mg, kind, k, v, q, chunk, capacity):
    """Prefill the whole history in chunks of `chunk` (append after each)."""
    B, T = k.shape[0], k.shape[1]
    cache = mg.KVCache(kind, B, capacity)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    outs = []
    kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
    for c0 in range(0, T, chunk):
        n = min(chunk, T - c0)
        kn, vn = kd[:, c0:c0 + n].contiguous(), vd[:, c0:c0 + n].contiguous()
        o, e = run_prefill(mg, kind, cache, [c0] * B, qd[:, c0:c0 + n], kn, vn, max_len=c0 + n)
        check_err(e)
        outs.append(o)
        mg.mg_kv_append(lay, cache, torch.tensor([c0] * B, dtype=torch.int32, device="cuda"), kn, vn,
                        err)
    torch.cuda.synchronize()
    check_err(err)
    return torch.cat(outs, dim=1)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("T,chunk", [(600, 600), (600, 256), (2600, 1000), (4500, 4500)])
def test_prefill_against_oracle(mg, kind, T, chunk):
    li = 2 if kind == 0 else 3
    k, v = synth.history(1, T, 21, li)
    q = synth.queries(1, T, 21, li)
    o = prefill_chunks(mg, kind, k, v, q, chunk, capacity=T)
    lay = orc.layer(oracle_kind(kind))
    rows = sorted(set(list(range(0, min(T, 40))) + list(range(T - 40, T)) +
                      list(range(0, T, max(1, T // 97)))))
    ref = orc.attention(lay, k[0], v[0], rows, q[0, rows])
    compare(o[0, rows], ref, f"kind {kind} T {T} chunk {chunk}")


@pytest.mark.parametrize("kind", [0, 1])
def test_chunked_equals_unchunked(mg, kind):
    T = 3000
    li = 2 if kind == 0 else 3
    k, v = synth.history(2, T, 22, li)
    q = synth.queries(2, T, 22, li)
    a = prefill_chunks(mg, kind, k, v, q, 3000, capacity=T)
    b = prefill_chunks(mg, kind, k, v, q, 512, capacity=T)
    d = (a.float() - b.float()).abs().max().item()
    assert d <= 2e-2, d


@pytest.mark.parametrize("kind", [0, 1])
def test_prefill_mixed_starts_with_a_rejected_sequence(mg, kind):
    # One call, three sequences: sequence 0 starts at 0, sequence 1's block
    # would run past max_len (flagged, its rows written as zeros), sequence 2
    # starts after 2500 cached positions (the local ring has wrapped).  1200
    # tokens make 150 query blocks per sequence and KV head.
    li = 2 if kind == 0 else 3
    B, n, c0s, max_len = 3, 1200, [0, 3000, 2500], 3700
    k, v = synth.history(B, 4200, 23, li)
    q = synth.queries(B, 4200, 23, li)
    cache = mg.KVCache(kind, B, max_len)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    mg.mg_kv_append(lay, cache, torch.tensor([-1, -1, 0], dtype=torch.int32, device="cuda"),
                    k[:, :2500].cuda().contiguous(), v[:, :2500].cuda().contiguous(), err)
    torch.cuda.synchronize()
    assert int(err.item()) & ~mg.DERR_POSITION == 0  # pos -1: the sequences left out
    qb = torch.stack([q[b, c0:c0 + n] for b, c0 in enumerate(c0s)])
    kb = torch.stack([k[b, c0:c0 + n] for b, c0 in enumerate(c0s)])
    vb = torch.stack([v[b, c0:c0 + n] for b, c0 in enumerate(c0s)])
    o, e = run_prefill(mg, kind, cache, c0s, qb, kb, vb, max_len)
    assert int(e.item()) == mg.DERR_POSITION, hex(int(e.item()))
    assert not o[1].float().abs().max().item()
    olay = orc.layer(oracle_kind(kind))
    for b in (0, 2):
        c0 = c0s[b]
        rows = sorted(set(list(range(0, 24)) + list(range(n - 24, n)) + list(range(0, n, 37))))
        pos = [c0 + i for i in rows]
        ref = orc.attention(olay, k[b, :c0 + n], v[b, :c0 + n], pos, q[b, pos])
        compare(o[b, rows], ref, f"kind {kind} sequence {b} c0 {c0}")
