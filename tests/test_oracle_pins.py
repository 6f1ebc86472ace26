"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test would fail under a plausible mistake in the oracle: a window off
by one, a wrong RoPE sign or pairing, a wrong KV-group map, a ring slot
formula error, a missing normalisation.  No GPU needed.

Sources: [P1] "深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？"
§01; [P2] "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
"窄缓存为长上下文留出空间" / "长上下文仍然带来计算开销"; [P4]
"Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析", "第二招".
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from hybrid_local_global_attn_b300 import synth

THETA = 10000.0
SCALE = 1.0 / math.sqrt(128.0)


def f64(x):
    return x.to(torch.float64).numpy()


def brute_force(kind, W, rope, k, v, qpos, q):
    """Explicit-matrix attention: dense score matrix, -inf mask, exp,
    normalise.  RoPE in complex form z = x[:64] + i x[64:], z *= e^{i t w}.
    Independent of the C oracle (different formulation, numpy)."""
    kd, vd, qd = f64(k), f64(v), f64(q)  # [T][2][128], [T][2][128], [nq][32][128]
    T = kd.shape[0]
    qpos = np.asarray(qpos)
    w = THETA ** (-2.0 * np.arange(64) / 128.0)

    def rot(x, t):
        z = (x[..., :64] + 1j * x[..., 64:]) * np.exp(1j * t[:, None, None] * w)
        return np.concatenate([z.real, z.imag], axis=-1)

    if rope:
        kd = rot(kd, np.arange(T, dtype=np.float64))
        qd = rot(qd, qpos.astype(np.float64))
    jj = np.arange(T)[None, :]
    pp = qpos[:, None]
    allowed = jj <= pp
    if kind == orc.LOCAL:
        allowed &= jj >= pp - W + 1
    mask = np.where(allowed, 0.0, -np.inf)  # [nq][T]
    out = np.zeros(qd.shape)
    for h in range(32):
        g = h // 16
        S = (qd[:, h, :] @ kd[:, g, :].T) * SCALE + mask
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ vd[:, g, :]
    return out


def rand_hist(T, seed):
    k = synth.randn_bf16((T, 2, 128), seed * 10 + 1)
    v = synth.randn_bf16((T, 2, 128), seed * 10 + 2)
    return k, v


@pytest.mark.parametrize("kind,W,rope", [(orc.LOCAL, 1, 1), (orc.LOCAL, 4, 1), (orc.LOCAL, 64, 1),
                                         (orc.LOCAL, 4, 0), (orc.GLOBAL, 0, 0), (orc.GLOBAL, 0, 1)])
def test_brute_force_tiny(kind, W, rope):
    T = 48
    k, v = rand_hist(T, 3)
    qpos = np.array([0, 1, 2, 3, 5, 17, 31, 46, 47], dtype=np.int32)
    q = synth.randn_bf16((len(qpos), 32, 128), 77)
    lay = orc.layer(kind, window=max(W, 1), rope=rope)
    got = orc.attention(lay, k, v, qpos, q)
    ref = brute_force(kind, W, rope, k, v, qpos, q)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_window_covering_history_is_rope_full_causal():
    # W >= T: a local layer equals full causal attention with RoPE [P1 §01]
    T = 200
    k, v = rand_hist(T, 5)
    qpos = np.arange(0, T, 7, dtype=np.int32)
    q = synth.randn_bf16((len(qpos), 32, 128), 8)
    a = orc.attention(orc.layer(orc.LOCAL, window=2048, rope=1), k, v, qpos, q)
    b = orc.attention(orc.layer(orc.GLOBAL, rope=1), k, v, qpos, q)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    # and it differs once the window is shorter than the history
    c = orc.attention(orc.layer(orc.LOCAL, window=64, rope=1), k, v, qpos, q)
    assert np.abs(c[-1] - a[-1]).max() > 1e-3


def test_rope_off_local_equals_global():
    # With RoPE switched off and W >= T, local and global compute the same set
    T = 150
    k, v = rand_hist(T, 6)
    qpos = np.arange(T, dtype=np.int32)
    q = synth.randn_bf16((T, 32, 128), 9)
    a = orc.attention(orc.layer(orc.LOCAL, window=2048, rope=0), k, v, qpos, q)
    b = orc.attention(orc.layer(orc.GLOBAL, rope=0), k, v, qpos, q)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kind", [orc.LOCAL, orc.GLOBAL])
def test_ring_cache_equals_linear_history(kind):
    # A 2048-slot ring that reuses the oldest slot [P2 窄缓存为长上下文留出空间]
    # plus the window mask gives the same outputs as the linear history.
    T = 2300
    k, v = rand_hist(T, 11)
    slots = 2048 if kind == orc.LOCAL else T
    kc = np.zeros((2, slots, 128), np.uint16)
    vc = np.zeros((2, slots, 128), np.uint16)
    lay = orc.layer(kind)
    # append in uneven pieces and decode the last appended position each
    # time: 999, 2046, 2047 (ring full), 2048 (first reuse), 2199, 2299
    cuts = [0, 1000, 2047, 2048, 2049, 2200, 2300]
    for a, b in zip(cuts[:-1], cuts[1:]):
        orc.cache_append(kind, kc, vc, a, k[a:b], v[a:b])
        p = b - 1
        q = synth.randn_bf16((32, 128), 1000 + p)
        got = orc.decode_from_cache(lay, kc, vc, p, q)
        ref = orc.attention(lay, k[:p + 1], v[:p + 1], [p], q.unsqueeze(0))[0]
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_cache_append_slots_bitwise():
    # local slot = pos mod 2048, global slot = pos; later positions overwrite
    T = 4200
    k, v = rand_hist(T, 12)
    kb = orc.bits(k)
    kc = np.zeros((2, 2048, 128), np.uint16)
    vc = np.zeros((2, 2048, 128), np.uint16)
    orc.cache_append(orc.LOCAL, kc, vc, 0, k[:3000], v[:3000])
    orc.cache_append(orc.LOCAL, kc, vc, 3000, k[3000:], v[3000:])
    for s in [0, 1, 103, 2047]:
        last = max(j for j in range(T) if j % 2048 == s)
        assert np.array_equal(kc[:, s, :], kb[last])
    gc = np.zeros((2, T, 128), np.uint16)
    gv = np.zeros((2, T, 128), np.uint16)
    orc.cache_append(orc.GLOBAL, gc, gv, 0, k, v)
    assert np.array_equal(gc.transpose(1, 0, 2), kb)
    with pytest.raises(ValueError):
        orc.cache_append(orc.GLOBAL, gc, gv, T, k[:1], v[:1])


@pytest.mark.parametrize("kind", [orc.LOCAL, orc.GLOBAL])
def test_commit_rolls_back_rejected_drafts(kind):
    # A speculative round [P4 第三招]: a 16-token block at p0 = 2040 (it
    # crosses the ring wrap) of which only the first 5 tokens are kept; the
    # other 11 are junk.  Afterwards the ring must still hold positions
    # p0 + i - 2048 for the rejected i (the slots the junk would have
    # reused), and decoding from the cache must equal attention over the
    # linear history of kept tokens, at the last kept position and after the
    # true continuation is appended.
    p0, n, keep, T = 2040, 16, 5, 2070
    k, v = rand_hist(T, 21)
    jk, jv = rand_hist(n, 22)  # junk drafts
    blk_k = torch.cat([k[p0:p0 + keep], jk[keep:]])
    blk_v = torch.cat([v[p0:p0 + keep], jv[keep:]])
    slots = 2048 if kind == orc.LOCAL else T
    kc = np.zeros((2, slots, 128), np.uint16)
    vc = np.zeros((2, slots, 128), np.uint16)
    orc.cache_append(kind, kc, vc, 0, k[:p0], v[:p0])
    orc.cache_commit(kind, kc, vc, p0, keep, blk_k, blk_v)
    kb = orc.bits(k)
    for i in range(keep, n):
        s = (p0 + i) % slots
        old = p0 + i - 2048  # the position a local slot held before the block
        want = kb[old] if kind == orc.LOCAL and old >= 0 else np.zeros_like(kb[0])
        assert np.array_equal(kc[:, s, :], want), f"rejected draft {i} reached slot {s}"
    lay = orc.layer(kind)
    for p in (p0 + keep - 1, T - 1):
        if p == T - 1:
            orc.cache_append(kind, kc, vc, p0 + keep, k[p0 + keep:], v[p0 + keep:])
        q = synth.randn_bf16((32, 128), 2000 + p)
        got = orc.decode_from_cache(lay, kc, vc, p, q)
        ref = orc.attention(lay, k[:p + 1], v[:p + 1], [p], q.unsqueeze(0))[0]
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # keeping nothing changes nothing; a count beyond the block is refused
    before = kc.copy()
    orc.cache_commit(kind, kc, vc, T, 0, blk_k, blk_v)
    assert np.array_equal(kc, before)
    with pytest.raises(ValueError):
        orc.cache_commit(kind, kc, vc, T, n + 1, blk_k, blk_v)


def test_paged_storage_map_worked_example_and_round_trip():
    # Page size 256, sequence 0 owns pages [5, 2, 7] and sequence 1 pages
    # [0, 3]: position 300 of sequence 0 is row 44 of page 2, position 700
    # row 188 of page 7; position 10 of sequence 1 row 10 of page 0.
    ps, pool = 256, 8
    kp = np.zeros((pool, 2, ps, 128), np.uint16)
    vp = np.zeros_like(kp)
    k0, v0 = rand_hist(701, 31)
    k1, v1 = rand_hist(300, 32)
    t0, t1 = [5, 2, 7], [0, 3]
    orc.paged_append(kp, vp, t0, ps, 0, k0[:301], v0[:301])  # two calls, the second
    orc.paged_append(kp, vp, t0, ps, 301, k0[301:], v0[301:])  # crossing a page
    orc.paged_append(kp, vp, t1, ps, 0, k1, v1)
    b0, b1 = orc.bits(k0), orc.bits(k1)
    assert np.array_equal(kp[2, :, 44], b0[300])
    assert np.array_equal(kp[7, :, 188], b0[700])
    assert np.array_equal(kp[0, :, 10], b1[10])
    assert np.array_equal(vp[3, :, 299 - 256], orc.bits(v1)[299])
    # pages nobody owns stay untouched
    for page in (1, 4, 6):
        assert not kp[page].any() and not vp[page].any()
    # reading back through the tables gives each linear history
    hk, hv = orc.paged_history(kp, vp, t0, ps, 701)
    assert np.array_equal(hk, b0) and np.array_equal(hv, orc.bits(v0))
    hk, hv = orc.paged_history(kp, vp, t1, ps, 300)
    assert np.array_equal(hk, b1)
    # attention over the paged history is attention over the linear one
    q = synth.randn_bf16((32, 128), 33)
    lay = orc.layer(orc.GLOBAL)
    hk, hv = orc.paged_history(kp, vp, t0, ps, 701)
    a = orc.attention(lay, hk, hv, [700], q.unsqueeze(0))
    b = orc.attention(lay, k0, v0, [700], q.unsqueeze(0))
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        orc.paged_append(kp, vp, [9], ps, 0, k1[:1], v1[:1])  # page outside the pool


def test_e4m3_codec_against_library_cast():
    # Every finite bf16 value, scaled by powers of two into and past the
    # e4m3 range: the oracle's round-to-nearest-even code equals torch's
    # float8_e4m3fn cast of the value clamped to +-448 (the saturation the
    # cache uses); decoding all 256 codes equals torch's widening.
    allbits = np.arange(65536, dtype=np.uint32)
    f32 = (allbits << 16).view(np.float32)
    f = f32[np.isfinite(f32)].astype(np.float64)
    for sc in (2.0 ** -8, 1.0, 2.0 ** 5):
        x = f * sc
        got = orc.e4m3_encode(x)
        want = torch.tensor(np.clip(x, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8)
        assert np.array_equal(got, want.numpy()), sc
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.e4m3_decode(codes), lib)


def test_e4m3_hand_values():
    # ties go to the even code, magnitudes past 448 saturate, the sign of
    # zero stays, subnormals step by 2^-9
    cases = {1.0: 0x38, 1.0625: 0x38, 1.1875: 0x3A, 1.9375: 0x40, 448.0: 0x7E, 500.0: 0x7E,
             -500.0: 0xFE, 2.0 ** -9: 0x01, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02,
             2.0 ** -6: 0x08, -1e-10: 0x80, 0.0: 0x00, -2.5: 0xC2}
    got = orc.e4m3_encode(np.array(list(cases)))
    assert got.tolist() == list(cases.values())
    assert orc.e4m3_decode(np.array([0x7F, 0xFF])).tolist().count(0) == 0  # NaN codes
    assert np.isnan(orc.e4m3_decode(np.array([0x7F]))[0])


def test_e4m3_cache_layout_and_round_trip():
    # V column order inside a 16-position group is a permutation; position 70
    # of head 1 sits in tile 1, column sigma(6) = 12; position 93 in column
    # 16 + sigma(13) = 27.  Values that are exact e4m3 multiples of the scale
    # come back bit for bit; others come back as the correctly rounded code.
    assert sorted(orc.E4M3_V_COLUMN) == list(range(16))
    assert orc.E4M3_V_COLUMN[6] == 12 and orc.E4M3_V_COLUMN[13] == 11
    T = 128
    kc = np.zeros((2, T, 128), np.uint8)
    vt = np.zeros((2, T // 64, 128, 64), np.uint8)
    ks, vs = [2.0 ** -2, 2.0], [1.0, 2.0 ** -3]
    vals = orc.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))  # finite, non-negative
    rng = np.random.default_rng(3)
    k = rng.choice(vals, size=(T, 2, 128)) * np.array(ks)[None, :, None]
    v = rng.choice(vals, size=(T, 2, 128)) * np.array(vs)[None, :, None]
    kb = torch.tensor(k, dtype=torch.float32).to(torch.bfloat16)
    vb = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16)
    orc.e4m3_cache_append(kc, vt, ks, vs, 0, kb[:70], vb[:70])
    orc.e4m3_cache_append(kc, vt, ks, vs, 70, kb[70:], vb[70:])
    assert np.array_equal(kc[1, 70], orc.e4m3_encode(k[70, 1] / ks[1]))
    assert np.array_equal(vt[1, 1, :, 12], orc.e4m3_encode(v[70, 1] / vs[1]))
    assert np.array_equal(vt[0, 1, :, 27], orc.e4m3_encode(v[93, 0] / vs[0]))
    hk, hv = orc.e4m3_history(kc, vt, ks, vs, T)
    assert np.array_equal(hk, orc.bits(kb)) and np.array_equal(hv, orc.bits(vb))
    # arbitrary bf16 inputs: the stored value is the nearest e4m3 multiple
    kr, vr = rand_hist(T, 41)
    orc.e4m3_cache_append(kc, vt, ks, vs, 0, kr, vr)
    hk, _ = orc.e4m3_history(kc, vt, ks, vs, T)
    x = f64(kr) / np.array(ks)[None, :, None]
    got = (hk.astype(np.uint32) << 16).view(np.float32).astype(np.float64) / np.array(ks)[None, :, None]
    err = np.abs(got - x)
    bound = np.maximum(np.ldexp(1.0, np.frexp(np.abs(x))[1] - 1 - 4), 2.0 ** -10)  # half a step
    assert np.all(err <= bound * (1 + 1e-12))
    with pytest.raises(ValueError):
        orc.e4m3_cache_append(kc, vt, [0.3, 1.0], vs, 0, kr[:1], vr[:1])


@pytest.mark.parametrize("kind,p", [(orc.LOCAL, 0), (orc.LOCAL, 100), (orc.LOCAL, 2046),
                                    (orc.LOCAL, 2047), (orc.LOCAL, 3000), (orc.GLOBAL, 3000)])
def test_zero_keys_give_window_mean(kind, p):
    # zero keys give equal scores whatever the rotation, so o is the mean of
    # V over exactly the key set: 2048 keys including the query itself for a
    # local layer [P1 §01], all p+1 keys for a global one.
    T = p + 1
    _, v = rand_hist(T, 13)
    k = torch.zeros((T, 2, 128), dtype=torch.bfloat16)
    q = synth.randn_bf16((1, 32, 128), 14)
    o = orc.attention(orc.layer(kind), k, v, [p], q)[0]
    lo = max(0, p - 2047) if kind == orc.LOCAL else 0
    vd = f64(v)
    for h in (0, 15, 16, 31):
        np.testing.assert_allclose(o[h], vd[lo:p + 1, h // 16].mean(axis=0), rtol=0, atol=1e-12)


def test_probability_rows_sum_to_one_and_respect_window():
    T = 3000
    k, _ = rand_hist(T, 15)
    q = synth.randn_bf16((128,), 16)
    for kind, p in [(orc.LOCAL, 2999), (orc.LOCAL, 10), (orc.GLOBAL, 2999)]:
        pr = orc.probs(orc.layer(kind), k, p, q, head=20)
        assert abs(pr.sum() - 1.0) < 1e-12
        lo = max(0, p - 2047) if kind == orc.LOCAL else 0
        assert (pr[:lo] == 0).all() and (pr[p + 1:] == 0).all()
        assert (pr[lo:p + 1] > 0).all()


def test_single_key_returns_its_value():
    k, v = rand_hist(1, 17)
    q = synth.randn_bf16((1, 32, 128), 18)
    for kind in (orc.LOCAL, orc.GLOBAL):
        o = orc.attention(orc.layer(kind), k, v, [0], q)[0]
        for h in range(32):
            np.testing.assert_allclose(o[h], f64(v)[0, h // 16], rtol=0, atol=0)


def test_two_keys_closed_form_with_rope():
    # q = a e0 at position 1; k0 = k1 = e0 at positions 0 and 1.
    # R(1) rotates (e0, e64) by angle w0 = 1 rad, so
    #   s0 = a cos(1) / sqrt(128),  s1 = a / sqrt(128),
    #   o  = sigmoid(s1 - s0) v1 + sigmoid(s0 - s1) v0.
    a = 8.0
    k = torch.zeros((2, 2, 128), dtype=torch.bfloat16)
    k[:, :, 0] = 1.0
    _, v = rand_hist(2, 19)
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16)
    q[0, :, 0] = a
    o = orc.attention(orc.layer(orc.LOCAL), k, v, [1], q)[0]
    s0 = a * math.cos(1.0) * SCALE
    s1 = a * SCALE
    w1 = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    vd = f64(v)
    for h in (0, 31):
        g = h // 16
        np.testing.assert_allclose(o[h], w1 * vd[1, g] + (1 - w1) * vd[0, g], rtol=0, atol=1e-13)


def test_one_hot_large_score_selects_value():
    T = 500
    _, v = rand_hist(T, 20)
    k = torch.zeros((T, 2, 128), dtype=torch.bfloat16)
    k[321, :, 5] = 64.0
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16)
    q[0, :, 5] = 64.0
    o = orc.attention(orc.layer(orc.GLOBAL), k, v, [499], q)[0]
    for h in (0, 17):
        np.testing.assert_allclose(o[h], f64(v)[321, h // 16], rtol=0, atol=1e-12)


def test_rope_identity_norm_composition_and_frequencies():
    x = np.random.default_rng(0).standard_normal(128)
    np.testing.assert_array_equal(orc.rope(x, 0.0), x)
    for t in (1.0, 37.0, 131071.0):
        np.testing.assert_allclose(np.linalg.norm(orc.rope(x, t)), np.linalg.norm(x), rtol=1e-14)
    np.testing.assert_allclose(orc.rope(orc.rope(x, 300.0), 45.0), orc.rope(x, 345.0), atol=1e-12)
    # rotate-half pairing: e_i goes to cos e_i + sin e_{i+64}, w_i = theta^(-2i/128)
    for i in (0, 1, 33, 63):
        e = np.zeros(128); e[i] = 1.0
        t = 5.0
        wi = THETA ** (-2.0 * i / 128.0)
        r = orc.rope(e, t)
        exp = np.zeros(128); exp[i] = math.cos(t * wi); exp[i + 64] = math.sin(t * wi)
        np.testing.assert_allclose(r, exp, atol=1e-15)


def test_local_outputs_invariant_to_position_shift():
    # RoPE makes scores depend on j - p only: shifting the whole local history
    # by D positions (padding in front, outside every window) leaves outputs equal.
    W, T, D = 64, 160, 1000
    k, v = rand_hist(T, 21)
    kp, vp = rand_hist(D, 22)
    qpos = np.arange(W, T, 9, dtype=np.int32)
    q = synth.randn_bf16((len(qpos), 32, 128), 23)
    lay = orc.layer(orc.LOCAL, window=W)
    a = orc.attention(lay, k, v, qpos, q)
    b = orc.attention(lay, torch.cat([kp, k]), torch.cat([vp, v]), qpos + D, q)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_query_head_reads_kv_group_h_div_16():
    # swapping the two KV heads and the two halves of the query heads swaps
    # the output halves: head h reads KV head h // 16 (not h % 2).
    T = 90
    k, v = rand_hist(T, 24)
    q = synth.randn_bf16((3, 32, 128), 25)
    pos = [10, 50, 89]
    for kind in (orc.LOCAL, orc.GLOBAL):
        lay = orc.layer(kind)
        a = orc.attention(lay, k, v, pos, q)
        b = orc.attention(lay, k.flip(1), v.flip(1), pos, torch.cat([q[:, 16:], q[:, :16]], 1))
        np.testing.assert_allclose(a[:, :16], b[:, 16:], atol=1e-13)
        np.testing.assert_allclose(a[:, 16:], b[:, :16], atol=1e-13)
        # identical queries within a group give identical outputs
        qq = q.clone(); qq[:, 1:16] = qq[:, :1]
        c = orc.attention(lay, k, v, pos, qq)
        assert np.array_equal(c[:, 0], c[:, 7])


def test_block_verify_equals_sequential_decodes():
    # a 16-token block attended in one pass with a causal mask inside the
    # block [P1 §04] equals 16 single-token decodes from a growing ring cache
    T0, n = 2040, 16
    k, v = rand_hist(T0 + n, 26)
    q = synth.randn_bf16((n, 32, 128), 27)
    for kind in (orc.LOCAL, orc.GLOBAL):
        lay = orc.layer(kind)
        block = orc.attention(lay, k, v, np.arange(T0, T0 + n, dtype=np.int32), q)
        slots = 2048 if kind == orc.LOCAL else T0 + n
        kc = np.zeros((2, slots, 128), np.uint16); vc = np.zeros_like(kc)
        orc.cache_append(kind, kc, vc, 0, k[:T0], v[:T0])
        for i in range(n):
            orc.cache_append(kind, kc, vc, T0 + i, k[T0 + i:T0 + i + 1], v[T0 + i:T0 + i + 1])
            d = orc.decode_from_cache(lay, kc, vc, T0 + i, q[i])
            np.testing.assert_allclose(block[i], d, rtol=0, atol=1e-12)


def test_full_attention_pair_count_matches_pages(golden_bytes):
    # about 1.7e10 attention computations per full layer at 131K [P4 第二招]: n^2
    val, tol, _ = golden_bytes["full_attention_pairs_131k"]
    n = 131072
    assert abs(n * n - val) <= tol * val


# --------------------------------------------------------------------------
# Peaked and flat score distributions: the inputs the GPU parity tests use to
# reach every softmax branch (queries scaled by 1e-3, 1, 40; a sink key far
# above the rest).  The oracle is pinned on the same kind of inputs here.

def brute_scores(kind, W, rope, k, qpos, q):
    """Scaled scores [nq][32][T] with -inf outside the key set, in numpy with
    complex-number RoPE (the formulation of brute_force above)."""
    kd, qd = f64(k), f64(q)
    T = kd.shape[0]
    qpos = np.asarray(qpos)
    w = THETA ** (-2.0 * np.arange(64) / 128.0)

    def rot(x, t):
        z = (x[..., :64] + 1j * x[..., 64:]) * np.exp(1j * t[:, None, None] * w)
        return np.concatenate([z.real, z.imag], axis=-1)

    if rope:
        kd = rot(kd, np.arange(T, dtype=np.float64))
        qd = rot(qd, qpos.astype(np.float64))
    jj = np.arange(T)[None, :]
    allowed = jj <= qpos[:, None]
    if kind == orc.LOCAL:
        allowed &= jj >= qpos[:, None] - W + 1
    s = np.einsum("nhd,tgd->nhtg", qd, kd)  # [nq][32][T][2]
    s = np.stack([s[:, h, :, h // 16] for h in range(32)], axis=1) * SCALE
    return np.where(allowed[:, None, :], s, -np.inf)


@pytest.mark.parametrize("kind", [orc.LOCAL, orc.GLOBAL])
@pytest.mark.parametrize("factor", [1e-3, 40.0, 400.0])
def test_scaled_queries_match_brute_force(kind, factor):
    # x400 puts scores near +-1e3: exp() of them overflows fp64 unless the
    # running maximum is subtracted first, so a softmax written without it
    # fails here; x1e-3 makes every row nearly uniform.
    T = 300
    k, v = rand_hist(T, 21)
    qpos = np.array([0, 1, 7, 63, 64, 150, 255, 256, 299], dtype=np.int32)
    q = synth.scaled(synth.randn_bf16((len(qpos), 32, 128), 22), factor)
    W = 100 if kind == orc.LOCAL else 0
    lay = orc.layer(kind, window=max(W, 1))
    got = orc.attention(lay, k, v, qpos, q)
    ref = brute_force(kind, W, kind == orc.LOCAL, k, v, qpos, q)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11)
    if factor == 1e-3:
        # nearly uniform: within 1e-2 of the mean of V over the key set
        for n, p in enumerate(qpos):
            lo = max(0, p - W + 1) if kind == orc.LOCAL else 0
            mean = f64(v[lo:p + 1]).mean(axis=0)  # [2][128]
            for h in range(32):
                assert np.abs(got[n, h] - mean[h // 16]).max() < 1e-2


@pytest.mark.parametrize("kind", [orc.LOCAL, orc.GLOBAL])
def test_sink_key_closed_form(kind):
    # A sink key scoring far above every other key: the output is that key's
    # value row up to (1 - P_sink) * max |v_j - v_sink|, with 1 - P_sink
    # bounded by sum_j exp(s_j - s_sink) (scores from the numpy formulation).
    T = 2600
    k, v = rand_hist(T, 23)
    sinks = [5, 2400]  # the later one scores ~22 above the earlier one
    k = synth.plant_sinks(k.unsqueeze(0), sinks, values=[synth.SINK_K, 1.5 * synth.SINK_K])[0]
    qpos = np.array([0, 4, 5, 6, 300, 2047, 2052, 2399, 2400, 2599], dtype=np.int32)
    q = synth.sink_queries(synth.randn_bf16((len(qpos), 32, 128), 24))
    W = 2048 if kind == orc.LOCAL else 0
    lay = orc.layer(kind)
    got = orc.attention(lay, k, v, qpos, q)
    s = brute_scores(kind, W, kind == orc.LOCAL, k, qpos, q)
    vd = f64(v)
    checked = 0
    for n, p in enumerate(qpos):
        visible = [j for j in sinks if j <= p and (kind == orc.GLOBAL or j > p - W)]
        if not visible:
            continue
        j = max(visible)  # the later sink also wins when both are visible
        for h in range(32):
            row = s[n, h]
            margin = row[j] - np.max(np.delete(row, j))
            assert margin > 20, (p, h, margin)
            tail = np.exp(np.delete(row, j) - row[j]).sum()
            bound = tail * np.abs(vd[:, h // 16] - vd[j, h // 16]).max() + 1e-12
            assert np.abs(got[n, h] - vd[j, h // 16]).max() <= bound
            checked += 1
    assert checked >= 7 * 32


# --------------------------------------------------------------------------
# QKV projection (hidden size 6656 -> 32 query heads + 2 key + 2 value heads
# of 128 [P1 §01]): y = x W^T in fp64, features laid out q | k | v.

def test_qkv_projection_selection_weights_pick_inputs():
    # W row f = e_{pi(f)}: every output is one input value, exactly, and the
    # q / k / v split puts feature 128 h + d of q head h, 4096 + 128 g + d of
    # key head g and 4352 + 128 g + d of value head g where the layout says.
    rng = np.random.default_rng(5)
    perm = rng.integers(0, orc.HIDDEN, size=orc.QKV_FEATURES)
    w = torch.zeros((orc.QKV_FEATURES, orc.HIDDEN), dtype=torch.bfloat16)
    w[torch.arange(orc.QKV_FEATURES), torch.from_numpy(perm)] = 1.0
    x = synth.randn_bf16((3, orc.HIDDEN), 61)
    y = orc.qkv_project(x, w)
    xd = f64(x)
    assert np.array_equal(y, xd[:, perm])
    q, k, v = orc.qkv_split(y)
    assert q.shape == (3, 32, 128) and k.shape == (3, 2, 128) and v.shape == (3, 2, 128)
    assert q[1, 5, 7] == xd[1, perm[128 * 5 + 7]]
    assert k[2, 1, 100] == xd[2, perm[4096 + 128 + 100]]
    assert v[0, 0, 3] == xd[0, perm[4352 + 3]]


def test_qkv_projection_matches_exact_sums():
    # against math.fsum (a correctly rounded sum of the exact products) on a
    # sample of outputs, and doubling x doubles y exactly
    x = synth.randn_bf16((2, orc.HIDDEN), 62)
    w = synth.scaled(synth.randn_bf16((orc.QKV_FEATURES, orc.HIDDEN), 63), 1.0 / 64)
    y = orc.qkv_project(x, w)
    xd, wd = f64(x), f64(w)
    for m in range(2):
        for f in [0, 1, 127, 128, 4095, 4096, 4351, 4352, 4607]:
            exact = math.fsum(xd[m] * wd[f])
            assert abs(y[m, f] - exact) <= 1e-12 * np.abs(xd[m] * wd[f]).sum()
    y2 = orc.qkv_project(synth.scaled(x, 2.0), w)
    assert np.array_equal(y2, 2 * y)


def test_qkv_fp32_accumulation_bound_holds():
    # the tolerance the GPU test uses: an fp32 sum of the 6656 products in
    # any order stays within gamma_6656 |x| |W|^T of the exact value
    # (checked here for sequential and pairwise fp32 orders)
    x = synth.randn_bf16((2, orc.HIDDEN), 64)
    w = synth.scaled(synth.randn_bf16((16, orc.HIDDEN), 65), 1.0 / 64)
    wfull = torch.zeros((orc.QKV_FEATURES, orc.HIDDEN), dtype=torch.bfloat16)
    wfull[:16] = w
    y = orc.qkv_project(x, wfull)[:, :16]
    bound = orc.FP32_GAMMA_HIDDEN * orc.qkv_abs_bound(x, wfull)[:, :16]
    prods = (f64(x)[:, None, :] * f64(w)[None, :, :]).astype(np.float32)  # exact in fp32
    seq = np.zeros((2, 16), np.float32)
    for i in range(orc.HIDDEN):
        seq += prods[:, :, i]
    pair = prods.sum(axis=2, dtype=np.float32)
    for s in (seq, pair):
        assert (np.abs(s.astype(np.float64) - y) <= bound).all()
    assert bound.max() < 0.05  # outputs here have sigma ~1.3
