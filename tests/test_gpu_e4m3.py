"""FP8 (e4m3) global-layer cache: codes compared bit for bit with the oracle's
store, decode against the fp64 oracle over the dequantised history (code x
power-of-two scale, the values the cache holds), so the tolerance covers the
kernel's arithmetic only ("Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳
Muse Glimmer", "窄缓存为长上下文留出空间": quantising the cache shrinks it)."""
import numpy as np
import pytest
import torch

from gpu_util import check_err, compare
from hybrid_local_global_attn_b300 import synth
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

GLOBAL = 1
KS, VS = (0.5, 2.0), (0.25, 1.0)


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def oracle_codes(B, slots, k, v, lengths, ks=KS, vs=VS):
    out = []
    for b, n in enumerate(lengths):
        kc = np.zeros((2, slots, 128), np.uint8)
        vt = np.zeros((2, slots // 64, 128, 64), np.uint8)
        if n:
            orc.e4m3_cache_append(kc, vt, ks, vs, 0, k[b, :n], v[b, :n])
        out.append((kc, vt))
    return out


def fill(mg, B, capacity, k, v, lengths, ks=KS, vs=VS):
    """FP8 cache holding positions [0, lengths[b]) of each sequence, appended
    through the library in two pieces."""
    cache = mg.E4M3KVCache(B, capacity, ks, vs)
    lay = mg.make_layer(GLOBAL)
    err = mg.error_word()
    for b, n in enumerate(lengths):
        cut = min(n, 333)
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
    torch.cuda.synchronize()
    assert int(err.item()) & ~mg.DERR_POSITION == 0  # pos -1 = the sequences left out
    return cache


def test_e4m3_append_and_commit_codes_bit_exact(mg):
    B, cap = 2, 1024
    lengths = [700, 129]
    k, v = synth.history(B, cap, 101, 3)
    # magnitudes past the e4m3 range saturate; tiny ones go subnormal or to 0
    k[0, 5, 0, :8] = torch.tensor([300, -300, 1e-3, -1e-3, 5e-4, 7, -7, 0], dtype=torch.bfloat16)
    v[1, 70, 1, :4] = torch.tensor([1000, -1000, 2e-3, -0.0], dtype=torch.bfloat16)
    cache = fill(mg, B, cap, k, v, lengths)
    want = oracle_codes(B, cache.slots, k, v, lengths)
    for b in range(B):
        assert np.array_equal(cache.k[b].cpu().numpy(), want[b][0]), f"K codes of sequence {b}"
        assert np.array_equal(cache.v[b].cpu().numpy(), want[b][1]), f"V codes of sequence {b}"
    # a commit of 5 and 16 of a 16-token block
    err = mg.error_word()
    p0 = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([5, 16], dtype=torch.int32, device="cuda")
    bk = torch.stack([k[b, n:n + 16] for b, n in enumerate(lengths)])
    bv = torch.stack([v[b, n:n + 16] for b, n in enumerate(lengths)])
    mg.mg_kv_commit(mg.make_layer(GLOBAL), cache, p0, cnt, bk.cuda().contiguous(),
                    bv.cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err)
    for b, n in enumerate(lengths):
        kc, vt = want[b]
        orc.e4m3_cache_append(kc, vt, KS, VS, n, bk[b, :int(cnt[b])], bv[b, :int(cnt[b])])
        assert np.array_equal(cache.k[b].cpu().numpy(), kc), f"K codes after commit, {b}"
        assert np.array_equal(cache.v[b].cpu().numpy(), vt), f"V codes after commit, {b}"


def oracle_decode(k, v, b, p, q_row, slots, ks=KS, vs=VS):
    kc = np.zeros((2, slots, 128), np.uint8)
    vt = np.zeros((2, slots // 64, 128, 64), np.uint8)
    orc.e4m3_cache_append(kc, vt, ks, vs, 0, k[b, :p + 1], v[b, :p + 1])
    hk, hv = orc.e4m3_history(kc, vt, ks, vs, p + 1)
    return orc.attention(orc.layer(orc.GLOBAL), hk, hv, [p], q_row)[0]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("positions", [[0, 63, 64], [700, 4095, 2222], [129, 5, 4000]])
def test_e4m3_decode_against_oracle(mg, positions, fused):
    B = len(positions)
    cap = max(positions) + 64
    k, v = synth.history(B, cap, 102, 3)
    q = synth.queries(B, 1, 102, 3)[:, 0]
    hist = positions if fused else [p + 1 for p in positions]
    cache = fill(mg, B, cap, k, v, hist)
    lay = mg.make_layer(GLOBAL)
    max_len = max(positions) + 1
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    err = mg.error_word()
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, max_len)
    if fused:
        kn = torch.stack([k[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
        vn = torch.stack([v[b, p:p + 1] for b, p in enumerate(positions)]).cuda().contiguous()
        mg.mg_append_decode(lay, cache, pos, max_len, q.cuda().contiguous(), kn, vn, o, ws, err)
    else:
        mg.mg_attn_decode(lay, cache, pos, max_len, q.cuda().contiguous(), o, ws, err)
    torch.cuda.synchronize()
    check_err(err)
    for b, p in enumerate(positions):
        ref = oracle_decode(k, v, b, p, q[b:b + 1], cache.slots)
        compare(o[b], ref, f"e4m3 decode b {b} p {p} fused {fused}")


def test_e4m3_decode_long_context_and_query_magnitudes(mg):
    # 131072 + 64 keys at batch 1 (148 splits), queries scaled down and up:
    # the kernel moves each query row to f16 with its own power of two
    B, cap = 1, 131072 + 64
    p = cap - 1
    k, v = synth.history(B, cap, 103, 3)
    cache = fill(mg, B, cap, k, v, [cap])
    kc = np.zeros((2, cache.slots, 128), np.uint8)
    vt = np.zeros((2, cache.slots // 64, 128, 64), np.uint8)
    orc.e4m3_cache_append(kc, vt, KS, VS, 0, k[0], v[0])
    hk, hv = orc.e4m3_history(kc, vt, KS, VS, p + 1)
    lay = mg.make_layer(GLOBAL)
    ws = mg.workspace(mg.OP_DECODE, lay, B, 1, cap)
    for qmul in (1e-3, 1.0, 40.0):
        q = (synth.queries(B, 1, 103, 3)[:, 0].float() * qmul).to(torch.bfloat16)
        o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
        err = mg.error_word()
        mg.mg_attn_decode(lay, cache, torch.tensor([p], dtype=torch.int32, device="cuda"), cap,
                          q.cuda().contiguous(), o, ws, err)
        torch.cuda.synchronize()
        check_err(err)
        ref = orc.attention(orc.layer(orc.GLOBAL), hk, hv, [p], q[:1])[0]
        compare(o[0], ref, f"e4m3 decode at {p}, query x {qmul}")
