"""KV append: cache contents bit-exact against the oracle's sequential replay
(local ring slot = pos mod 2048, global slot = pos)."""
import numpy as np
import pytest
import torch

from gpu_util import bits_of, cache_expected, check_err
from hybrid_local_global_attn_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import mg as m
    return m


def run_appends(mg, kind, B, capacity, T, appends, seed):
    """appends: list of (pos0 per sequence list, n).  Returns GPU cache + histories."""
    k, v = synth.history(B, T, seed, 0)
    cache = mg.KVCache(kind, B, capacity)
    lay = mg.make_layer(kind)
    err = mg.error_word()
    kd, vd = k.cuda(), v.cuda()
    per_seq = [[] for _ in range(B)]
    for pos0s, n in appends:
        kn = torch.stack([kd[b, p:p + n] for b, p in enumerate(pos0s)]).contiguous()
        vn = torch.stack([vd[b, p:p + n] for b, p in enumerate(pos0s)]).contiguous()
        pos = torch.tensor(pos0s, dtype=torch.int32, device="cuda")
        mg.mg_kv_append(lay, cache, pos, kn, vn, err)
        for b, p in enumerate(pos0s):
            per_seq[b].append((p, n))
    torch.cuda.synchronize()
    return cache, k, v, per_seq, err


@pytest.mark.parametrize("kind", [0, 1])
def test_append_bitexact_mixed(mg, kind):
    B, T = 3, 6000
    cap = T
    appends = [([0, 0, 0], 1), ([1, 1, 1], 2047), ([2048, 2048, 2048], 1),  # fill, then wrap
               ([2049, 2100, 3000], 5), ([2054, 2105, 3005], 2500)]          # ragged, n > 2048
    cache, k, v, per_seq, err = run_appends(mg, kind, B, cap, T, appends, seed=3)
    check_err(err)
    for b in range(B):
        kc, vc = cache_expected(kind, cache.slots, k[b], v[b], per_seq[b])
        assert np.array_equal(bits_of(cache.k[b]), kc), f"K sequence {b}"
        assert np.array_equal(bits_of(cache.v[b]), vc), f"V sequence {b}"


def test_append_single_tokens_across_wrap(mg):
    T = 2100
    appends = [([0], 2040)] + [([p], 1) for p in range(2040, 2100)]
    cache, k, v, per_seq, err = run_appends(mg, 0, 1, 0, T, appends, seed=4)
    check_err(err)
    kc, vc = cache_expected(0, 2048, k[0], v[0], per_seq[0])
    assert np.array_equal(bits_of(cache.k[0]), kc)
    assert np.array_equal(bits_of(cache.v[0]), vc)


def test_append_past_global_capacity_flags_and_skips(mg):
    B, cap = 2, 100
    k, v = synth.history(B, 110, 5, 0)
    cache = mg.KVCache(1, B, cap)
    lay = mg.make_layer(1)
    err = mg.error_word()
    pos = torch.tensor([90, 10], dtype=torch.int32, device="cuda")
    mg.mg_kv_append(lay, cache, pos, k[:, :20].cuda().contiguous(), v[:, :20].cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err, mg.DERR_POSITION)
    kb = bits_of(cache.k)
    kh = bits_of(k)
    # sequence 0: positions 90..99 written, 100..109 skipped
    assert np.array_equal(kb[0][:, 90:100].transpose(1, 0, 2), kh[0][0:10])
    # sequence 1 unaffected: 10..29
    assert np.array_equal(kb[1][:, 10:30].transpose(1, 0, 2), kh[1][0:20])
    # negative position: flagged, nothing written
    err.zero_()
    c2 = mg.KVCache(0, 1)
    mg.mg_kv_append(mg.make_layer(0), c2, torch.tensor([-3], dtype=torch.int32, device="cuda"),
                    k[:1, :4].cuda().contiguous(), v[:1, :4].cuda().contiguous(), err)
    torch.cuda.synchronize()
    check_err(err, mg.DERR_POSITION)
    assert int(c2.k.abs().sum().item()) == 0
