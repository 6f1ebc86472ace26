"""mg_attn_decode_noalloc: decode for callers that cannot allocate device
memory (a plugin whose host framework owns all device buffers, or a serving
loop that must not call cudaMalloc).  Its split partials live in a fixed
array inside libmg.so instead of a caller workspace.

Checked here, through the C ABI, on two calls in a row: the outputs equal,
bit for bit, those of mg_attn_decode with a caller-allocated workspace (both
run the same kernels with the same split count, so any difference -- a stale
partial left in the shared array by the previous call, say -- shows), and
they match the fp64 oracle within the parity tolerance.  The cases cover a
mixed batch (49 splits, the row combine) and batch 1 at a long context (148
splits, the wide combine), the case that uses the most of the array.  That
every batch fits the fixed array is a host-side check in test_abi.py.  The
file is collected last so that a run stopping at the first failure has run
every other test.
"""
import ctypes

import pytest
import torch

from gpu_util import check_err, compare, oracle_kind
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    f = m.lib.mg_attn_decode_noalloc
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(m.mg_layer), ctypes.POINTER(m.mg_cache), P, ctypes.c_int32, P, P,
                  P, P]
    f.restype = ctypes.c_int
    return m


@pytest.mark.parametrize("kind,positions,T", [
    (0, [4999, 2047, 130], 5000),
    (1, [4999, 2047, 130], 5000),
    (1, [131135], 131136),  # batch 1, 148 splits: the largest use of the array
])
def test_noalloc_decode_matches_workspace_decode(mg, kind, positions, T):
    B = len(positions)
    li = 3 if kind == 1 else 2
    k, v = synth.history(B, T, 31, li)
    q = synth.queries(B, 1, 31, li)[:, 0].cuda().contiguous()
    cache = mg.KVCache(kind, B, T)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    if kind == 1:
        pos0, n = [0] * B, T
    else:
        pos0, n = [max(0, p - 2047) for p in positions], 2048
    kn = torch.stack([k[b, p:p + n] for b, p in enumerate(pos0)]).cuda().contiguous()
    vn = torch.stack([v[b, p:p + n] for b, p in enumerate(pos0)]).cuda().contiguous()
    mg.mg_kv_append(lay, cache, torch.tensor(pos0, dtype=torch.int32, device="cuda"), kn, vn, err)
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    max_len = max(positions) + 1

    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, max_len)
    o_ref = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    mg.mg_attn_decode(lay, cache, pos, max_len, q, o_ref, ws, err)
    torch.cuda.synchronize()
    check_err(err)

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        o = torch.full((B, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = mg.lib.mg_attn_decode_noalloc(ctypes.byref(lay), ctypes.byref(cache.struct),
                                           ctypes.c_void_p(pos.data_ptr()), max_len,
                                           ctypes.c_void_p(q.data_ptr()),
                                           ctypes.c_void_p(o.data_ptr()),
                                           ctypes.c_void_p(err.data_ptr()), stream)
        assert rc == 0, mg.mg_status_str(rc)
        torch.cuda.synchronize()
        check_err(err)
        assert torch.equal(o, o_ref), (
            f"kind {kind} call {call}: differs from the workspace decode by "
            f"{(o.float() - o_ref.float()).abs().max().item()}")

    olay = orc.layer(oracle_kind(kind))
    qc = q.cpu()
    for b, p in enumerate(positions):
        ref = orc.attention(olay, k[b, :p + 1], v[b, :p + 1], [p], qc[b:b + 1])[0]
        compare(o[b], ref, f"kind {kind} b {b} p {p}")
