"""CPU checks of the C ABI: the library loads, exports every declared symbol,
its byte model matches the figures the pages print, and host-side argument
checks reject bad calls before touching CUDA.  No GPU needed.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mg.h")
GIB = 1024 ** 3
MIB = 1024 ** 2


@pytest.fixture(scope="module")
def mg():
    from hybrid_local_global_attn_b300 import build
    build.build()
    from hybrid_local_global_attn_b300 import mg as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mg_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(mg):
    names = declared_functions()
    assert {"mg_kv_append", "mg_attn_decode", "mg_attn_verify", "mg_attn_prefill",
            "mg_cache_bytes", "mg_workspace_bytes", "mg_status_str"} <= set(names)
    for n in names:
        assert hasattr(mg.lib, n), n
        assert ctypes.cast(getattr(mg.lib, n), ctypes.c_void_p).value


def test_binding_constants_match_header(mg):
    """The binding's flag, kind and op constants equal the header's #defines
    (a mismatch would pass the wrong bits through the C ABI)."""
    text = open(HEADER).read()
    defines = {k: int(v.rstrip("uU"), 0) for k, v in
               re.findall(r"#define\s+(MG_\w+)\s+(0x[0-9a-fA-F]+[uU]?|\d+[uU]?)\b", text)}
    assert defines["MG_EARLY_START"] == mg.EARLY_START == 1
    assert defines["MG_OVERLAP_NEXT"] == mg.OVERLAP_NEXT == 2
    assert mg.EARLY_START & mg.OVERLAP_NEXT == 0


def test_byte_model_matches_pages(mg, golden_bytes):
    gb = golden_bytes
    per_tok = mg.mg_cache_bytes(mg.GLOBAL, 1, 1)
    assert per_tok == gb["kv_bytes_per_token_layer"][0] == 1024
    T = 131072
    kinds = [mg.mg_layer_kind(l) for l in range(52)]
    assert kinds.count(mg.GLOBAL) == 13 and kinds.count(mg.LOCAL) == 39
    assert all((k == mg.GLOBAL) == (l % 4 == 3) for l, k in enumerate(kinds))
    glob = sum(mg.mg_cache_bytes(k, 1, T) for k in kinds if k == mg.GLOBAL)
    loc = sum(mg.mg_cache_bytes(k, 1, T) for k in kinds if k == mg.LOCAL)
    assert glob / GIB == gb["global_kv_gib"][0]          # 1.625 GiB exactly
    v, tol, _ = gb["local_kv_mib"]
    assert abs(loc / MIB - v) <= tol * v                  # 78 MiB
    v, tol, _ = gb["hybrid_kv_gib"]
    assert abs((glob + loc) / GIB - v) <= tol * v         # ~1.70 GiB
    v, tol, _ = gb["all_global_kv_gib"]
    allg = 52 * mg.mg_cache_bytes(mg.GLOBAL, 1, T)
    assert abs(allg / GIB - v) <= tol * v                 # 6.5 GiB
    # MHA: 32 KV heads instead of 2
    assert 32 // mg.HKV == gb["mha_factor"][0]
    assert (glob + loc) * 16 / GIB > gb["mha_kv_gib_at_least"][0]
    assert mg.mg_cache_bytes(mg.LOCAL, 3, 999999) == 3 * mg.mg_cache_bytes(mg.LOCAL, 1, 0)
    assert mg.mg_cache_bytes(7, 1, 10) == 0 and mg.mg_cache_bytes(mg.GLOBAL, 1, -1) == 0


def test_status_strings_and_kinds(mg):
    assert mg.mg_status_str(0) == "ok"
    for s in range(1, 6):
        assert mg.mg_status_str(s) not in ("ok", "unknown status")
    assert mg.mg_layer_kind(-1) == -1 and mg.mg_layer_kind(52) == -1


def test_workspace_sizes(mg):
    L = mg.make_layer(mg.LOCAL)
    G = mg.make_layer(mg.GLOBAL)
    for op, n in ((mg.OP_DECODE, 1), (mg.OP_VERIFY, 16), (mg.OP_PREFILL, 4096)):
        for lay in (L, G):
            w = mg.mg_workspace_bytes(op, lay, 2, n, 40000)
            assert w >= 0
    assert mg.mg_workspace_bytes(mg.OP_PREFILL, G, 1, 4096, 32768) == 0  # global prefill: none
    assert mg.mg_workspace_bytes(mg.OP_DECODE, G, 1, 1, 131073) > 0
    with pytest.raises(mg.MgError):
        mg.mg_workspace_bytes(mg.OP_VERIFY, G, 1, 17, 1000)     # block > 16
    with pytest.raises(mg.MgError):
        mg.mg_workspace_bytes(mg.OP_DECODE, G, 0, 1, 1000)      # batch 0
    bad = mg.mg_layer(mg.LOCAL, 1024, 1e4, mg.SCALE)             # window != 2048
    with pytest.raises(mg.MgError):
        mg.mg_workspace_bytes(mg.OP_DECODE, bad, 1, 1, 100)


def _raw_call_status(mg, fn, *args):
    return fn(*args)


def test_host_side_rejections_launch_nothing(mg):
    """Bad arguments come back as a status before any CUDA call (so this runs
    without a GPU).  Pointers are fake but never dereferenced on the host."""
    lib = mg.lib
    fake = ctypes.c_void_p(0x1000)
    cache = mg.mg_cache(0x10000, 0x20000, 1, 2048)
    L = mg.make_layer(mg.LOCAL)
    G = mg.make_layer(mg.GLOBAL)
    by = ctypes.byref
    # null layer / cache / positions
    assert lib.mg_kv_append(None, by(cache), fake, 1, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(L), None, fake, 1, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(L), by(cache), None, 1, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(L), by(cache), fake, -1, fake, fake, fake, None) == 1
    # n == 0 is a no-op
    assert lib.mg_kv_append(by(L), by(cache), fake, 0, fake, fake, fake, None) == 0
    # commit: counts are required; the next-position output must not alias pos0
    other = ctypes.c_void_p(0x3000)
    assert lib.mg_kv_commit(by(L), by(cache), fake, 4, None, fake, fake, None, fake, None) == 1
    assert lib.mg_kv_commit(by(L), by(cache), fake, 4, other, fake, fake, fake, fake, None) == 1
    assert lib.mg_kv_commit(by(L), by(cache), fake, -1, other, fake, fake, None, fake, None) == 1
    assert lib.mg_kv_commit(by(L), by(cache), fake, 4, other, ctypes.c_void_p(0x1008), fake,
                            None, fake, None) == 1
    assert lib.mg_kv_commit(by(L), by(cache), fake, 0, other, fake, fake, None, fake, None) == 0
    # FP8 caches: global, linear, 64-multiple slots, power-of-two scales;
    # verify and prefill take none
    def e4(slots, ks=(1.0, 0.5), vs=(2.0, 1.0), table=None):
        return mg.mg_cache(0x10000, 0x20000, 1, slots, table, 256 if table else 0, 4 if table else 0,
                           mg.E4M3, (ctypes.c_float * 2)(*ks), (ctypes.c_float * 2)(*vs))
    assert lib.mg_kv_append(by(L), by(e4(2048)), fake, 0, fake, fake, fake, None) == 2
    assert lib.mg_kv_append(by(G), by(e4(4096, ks=(0.3, 1.0))), fake, 0, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(G), by(e4(4096, vs=(0.0, 1.0))), fake, 0, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(G), by(e4(4000)), fake, 0, fake, fake, fake, None) == 1
    assert lib.mg_kv_append(by(G), by(e4(4096, table=0x3000)), fake, 0, fake, fake, fake, None) == 2
    assert lib.mg_kv_append(by(G), by(e4(4096)), fake, 0, fake, fake, fake, None) == 0
    assert lib.mg_attn_verify(by(G), by(e4(4096)), fake, 16, 1000, fake, fake, fake, fake, fake,
                              1 << 30, fake, None) == 2
    assert lib.mg_attn_prefill(by(G), by(e4(4096)), fake, 16, 1000, fake, fake, fake, fake, fake,
                               1 << 30, fake, None) == 2
    assert mg.mg_e4m3_cache_bytes(2, 4096) == 2 * 2 * 2 * 4096 * 128
    assert mg.mg_e4m3_cache_bytes(2, 4000) == 0
    # multi-layer commit: layer count in [1, 64], one batch for all caches
    lays = (mg.mg_layer * 2)(L, G)
    gcache = mg.mg_cache(0x10000, 0x20000, 1, 4096)
    caches = (mg.mg_cache * 2)(cache, gcache)
    for nl in (0, 65):
        assert lib.mg_kv_commit_layers(nl, lays, caches, fake, 4, other, fake, fake, None, fake,
                                       None) == 1
    caches2 = (mg.mg_cache * 2)(cache, mg.mg_cache(0x10000, 0x20000, 2, 4096))
    assert lib.mg_kv_commit_layers(2, lays, caches2, fake, 4, other, fake, fake, None, fake,
                                   None) == 1
    caches3 = (mg.mg_cache * 2)(gcache, gcache)  # local layer on a 4096-slot cache
    assert lib.mg_kv_commit_layers(2, lays, caches3, fake, 4, other, fake, fake, None, fake,
                                   None) == 2
    # local layer with a cache that is not a 2048-slot ring
    c2 = mg.mg_cache(0x10000, 0x20000, 1, 4096)
    assert lib.mg_kv_append(by(L), by(c2), fake, 1, fake, fake, fake, None) == 2
    # window / theta / scale out of range
    for bad in (mg.mg_layer(mg.LOCAL, 4096, 1e4, mg.SCALE), mg.mg_layer(mg.LOCAL, 2048, 0.0, mg.SCALE),
                mg.mg_layer(mg.GLOBAL, 2048, 0.0, mg.SCALE), mg.mg_layer(mg.GLOBAL, 0, 0.0, -1.0),
                mg.mg_layer(5, 0, 0.0, mg.SCALE)):
        assert lib.mg_attn_decode(by(bad), by(cache), fake, 10, fake, fake, fake, 1 << 30,
                                  fake, None) in (1, 2)
    # mg_append_decode_ex: unknown flag bits, and the checks of mg_append_decode
    gc = mg.mg_cache(0x10000, 0x20000, 1, 1000)
    for unknown in (4, 8 | mg.EARLY_START, 1 << 31):
        assert lib.mg_append_decode_ex(by(G), by(gc), fake, 1000, fake, fake, fake, fake, fake,
                                       1 << 30, fake, unknown, None) == 1
    for flags in (mg.EARLY_START, mg.OVERLAP_NEXT, mg.EARLY_START | mg.OVERLAP_NEXT):
        assert lib.mg_append_decode_ex(by(G), by(gc), fake, 1001, fake, fake, fake, fake, fake,
                                       1 << 30, fake, flags, None) == 3
        assert lib.mg_append_decode_ex(by(G), by(gc), fake, 1000, fake, None, fake, fake, fake,
                                       1 << 30, fake, flags, None) == 1
    # global decode past capacity
    assert lib.mg_attn_decode(by(G), by(gc), fake, 1001, fake, fake, fake, 1 << 30, fake, None) == 3
    # workspace too small
    need = mg.mg_workspace_bytes(mg.OP_DECODE, G, 1, 1, 1000)
    assert lib.mg_attn_decode(by(G), by(gc), fake, 1000, fake, fake, fake, need - 1, fake, None) == 4
    # misaligned tensor pointer
    assert lib.mg_attn_decode(by(G), by(gc), fake, 1000, ctypes.c_void_p(0x1002), fake, fake,
                              1 << 30, fake, None) == 1
    # verify block longer than 16
    assert lib.mg_attn_verify(by(G), by(gc), fake, 17, 1017, fake, fake, fake, fake, fake, 1 << 30,
                              fake, None) == 2
    # verify / prefill: cache too short for the positions before the block
    assert lib.mg_attn_prefill(by(G), by(gc), fake, 100, 1101, fake, fake, fake, fake, fake, 1 << 30,
                               fake, None) == 3
    assert lib.mg_attn_prefill(by(G), by(gc), fake, 0, 10, fake, fake, fake, fake, fake, 1 << 30,
                               fake, None) == 1


def test_noalloc_scratch_covers_every_decode_batch(mg):
    """The fixed array behind mg_attn_decode_noalloc (4 MiB) holds the decode
    workspace of any batch at the longest context: one split per KV head
    needs none, and the split count keeps splits x batch near 148."""
    lay = mg.make_layer(mg.GLOBAL)
    for B in list(range(1, 160)) + [256, 512, 4096]:
        for max_len in (1, 4096, 131072, 1 << 20):
            need = mg.mg_workspace_bytes(mg.OP_DECODE, lay, B, 1, max_len)
            assert need <= 4 << 20, (B, max_len, need)


def test_qkv_append_host_checks(mg):
    """mg_qkv_append: workspace sizes and argument checks, before any CUDA call."""
    lib = mg.lib
    by = ctypes.byref
    fake = ctypes.c_void_p(0x1000)
    # few tokens: the K range is split and fp32 partials need room; a full
    # grid of output tiles needs none
    assert mg.mg_qkv_workspace_bytes(1, 1) == 8 * 1 * mg.QKV_FEATURES * 4
    assert mg.mg_qkv_workspace_bytes(4, 40) == 4 * 160 * mg.QKV_FEATURES * 4  # 36 tiles, 4 splits
    assert mg.mg_qkv_workspace_bytes(1, 8192) == 0
    with pytest.raises(mg.MgError):
        mg.mg_qkv_workspace_bytes(0, 1)
    L, G = mg.make_layer(mg.LOCAL), mg.make_layer(mg.GLOBAL)
    ring = mg.mg_cache(0x10000, 0x20000, 1, 2048)
    args = lambda lay, c, n=1, x=fake, q=fake, k=None, v=None, ws=fake, wsb=1 << 30: (
        by(lay), by(c), fake, n, x, fake, q, k, v, ws, wsb, fake, None)
    assert lib.mg_qkv_append(*args(L, ring, x=None)) == 1             # no input
    assert lib.mg_qkv_append(*args(L, ring, q=None)) == 1             # no query output
    assert lib.mg_qkv_append(*args(L, ring, k=fake)) == 1             # k_out without v_out
    assert lib.mg_qkv_append(*args(L, ring, n=0)) == 1
    assert lib.mg_qkv_append(*args(L, ring, x=ctypes.c_void_p(0x1008))) == 1  # misaligned
    assert lib.mg_qkv_append(*args(L, ring, wsb=100)) == 4            # workspace too small
    e4 = mg.mg_cache(0x10000, 0x20000, 1, 4096, None, 0, 0, mg.E4M3,
                     (ctypes.c_float * 2)(1.0, 1.0), (ctypes.c_float * 2)(1.0, 1.0))
    assert lib.mg_qkv_append(*args(G, e4)) == 2                       # FP8 cache
    assert lib.mg_qkv_append(*args(L, mg.mg_cache(0x10000, 0x20000, 1, 4096))) == 2  # not a ring
