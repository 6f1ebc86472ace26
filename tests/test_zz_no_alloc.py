"""mg_attn_decode_noalloc: decode for callers that cannot allocate device
memory (a plugin whose host framework owns all device buffers, or a serving
loop that must not call cudaMalloc).  Its split partials live in a fixed
array inside libmg.so instead of a caller workspace.

Checked here, through the C ABI: two calls in a row give the same outputs
as mg_attn_decode with a caller-allocated workspace, within the parity
tolerance used by the other GPU tests.  That every batch fits the fixed
array is a host-side check in test_abi.py.  The file is
collected last so that a run stopping at the first failure has run every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import MAX_ABS, REL_L2, check_err
from hybrid_local_global_attn_b300 import synth

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


def close(a, b, what):
    x = a.float().cpu().double().numpy()
    y = b.float().cpu().double().numpy()
    err = np.abs(x - y).max()
    rel = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


@pytest.mark.parametrize("kind", [0, 1])
def test_noalloc_decode_matches_workspace_decode(mg, kind):
    B, T = 3, 5000
    positions = [4999, 2047, 130]
    k, v = synth.history(B, T, 31, 3 if kind == 1 else 2)
    q = synth.queries(B, 1, 31, 3 if kind == 1 else 2)[:, 0].cuda().contiguous()
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
        close(o, o_ref, f"kind {kind} call {call}")
