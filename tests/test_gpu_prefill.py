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
