"""Failure detection on the GPU without a fault: every pipeline wait in the
kernels is bounded, and a wait that runs out reports MG_DERR_TIMEOUT in the
caller's error word and lets the kernel return.

mg_debug_decode_stall runs a global-layer decode whose TMA producer stops
issuing key tiles at a chosen tile, so the consumers wait for a tile that
never arrives (a flag nothing sets).  With the wait limit lowered for that
call, the test sees the timeout come back quickly, and then checks that the
context is still usable: the ordinary decode on the same cache afterwards
matches the oracle."""
import time

import pytest
import torch

from gpu_util import check_err, compare
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


@pytest.mark.parametrize("stall_tile", [0, 2])
def test_stalled_producer_times_out_and_context_survives(mg, stall_tile):
    B, T = 1, 20000
    k, v = synth.history(B, T, 51, 3)
    q = synth.queries(B, 1, 51, 3)[:, 0]
    cache = mg.KVCache(mg.GLOBAL, B, T)
    lay = mg.make_layer(mg.GLOBAL)
    err = mg.error_word()
    mg.mg_kv_append(lay, cache, torch.tensor([0], dtype=torch.int32, device="cuda"),
                    k.cuda().contiguous(), v.cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err)
    p = T - 1
    pos = torch.tensor([p], dtype=torch.int32, device="cuda")
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, T)
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    qd = q.cuda().contiguous()

    t0 = time.perf_counter()
    mg.mg_debug_decode_stall(lay, cache, pos, T, qd, o, ws, err, wait_ns=2_000_000,
                             stall_tile=stall_tile)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(err.item()) == mg.DERR_TIMEOUT, hex(int(err.item()))
    assert took < 1.0, f"the stalled call took {took:.3f} s"  # 2 ms limit, not the 2 s default

    # the context still works: a normal decode of the same cache is correct
    err.zero_()
    mg.mg_attn_decode(lay, cache, pos, T, qd, o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    ref = orc.attention(orc.layer(orc.GLOBAL), k[0], v[0], [p], q)[0]
    compare(o[0], ref, "decode after a timed-out call")


def test_stall_entry_rejects_what_it_does_not_cover(mg):
    lay = mg.make_layer(mg.LOCAL)
    cache = mg.KVCache(mg.LOCAL, 1, 2048)
    pos = torch.tensor([10], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    err = mg.error_word()
    with pytest.raises(mg.MgError) as e:
        mg.mg_debug_decode_stall(lay, cache, pos, 11, q, o, None, err, wait_ns=1000, stall_tile=0)
    assert e.value.status == 2  # MG_ERR_UNSUPPORTED
