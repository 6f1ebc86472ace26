"""ctypes front end of the fp64 C oracle (``mg_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Arrays cross as numpy: bf16 tensors travel as
their raw ``uint16`` bit patterns, results come back as float64.  The C side
states which page passage each function follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

LOCAL = 0
GLOBAL = 1
HQ, HKV, D = 32, 2, 128
WINDOW = 2048
THETA = 10000.0
SCALE = 1.0 / np.sqrt(128.0)


class _Layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("rope", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("theta", ctypes.c_double), ("scale", ctypes.c_double)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        _lib.mg_oracle_attention.argtypes = [ctypes.POINTER(_Layer), i32, P, P, i32, P, P, P]
        _lib.mg_oracle_probs.argtypes = [ctypes.POINTER(_Layer), i32, P, i32, P, i32, P]
        _lib.mg_oracle_cache_append.argtypes = [i32, i32, P, P, i32, i32, P, P]
        _lib.mg_oracle_decode_from_cache.argtypes = [ctypes.POINTER(_Layer), i32, P, P, i32, P, P]
        _lib.mg_oracle_rope.argtypes = [P, ctypes.c_double, ctypes.c_double]
        _lib.mg_oracle_rope.restype = None
        _lib.mg_oracle_threads.restype = ctypes.c_int
    return _lib


def threads() -> int:
    return int(lib().mg_oracle_threads())


def layer(kind, window=WINDOW, rope=None, theta=THETA, scale=SCALE):
    """Oracle layer record.  RoPE defaults to on for local, off for global."""
    if rope is None:
        rope = 1 if kind == LOCAL else 0
    return _Layer(int(kind), int(window), int(rope), 0, float(theta), float(scale))


def bits(x) -> np.ndarray:
    """bf16 torch tensor (or uint16 array) -> contiguous uint16 numpy bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(lay, k_hist, v_hist, q_pos, q):
    """o[nq][32][128] (float64) for queries at q_pos against history [T][2][128]."""
    k = bits(k_hist); v = bits(v_hist); qq = bits(q)
    T = k.shape[0]
    assert k.shape == (T, HKV, D) and v.shape == (T, HKV, D)
    pos = np.ascontiguousarray(np.asarray(q_pos, dtype=np.int32))
    nq = pos.shape[0]
    assert qq.shape == (nq, HQ, D), qq.shape
    o = np.zeros((nq, HQ, D), dtype=np.float64)
    rc = lib().mg_oracle_attention(ctypes.byref(lay), T, _ptr(k), _ptr(v), nq,
                                   _ptr(pos), _ptr(qq), _ptr(o))
    if rc != 0:
        raise ValueError(f"mg_oracle_attention failed: {rc}")
    return o


def probs(lay, k_hist, p, q_row, head):
    k = bits(k_hist); qq = bits(q_row)
    T = k.shape[0]
    out = np.zeros(T, dtype=np.float64)
    rc = lib().mg_oracle_probs(ctypes.byref(lay), T, _ptr(k), int(p), _ptr(qq), int(head), _ptr(out))
    if rc != 0:
        raise ValueError(f"mg_oracle_probs failed: {rc}")
    return out


def cache_append(kind, k_cache, v_cache, pos0, k_new, v_new):
    """Replay appends into one sequence's cache ([2][slots][128] uint16, in place)."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    slots = k_cache.shape[1]
    kn = bits(k_new); vn = bits(v_new)
    n = kn.shape[0]
    rc = lib().mg_oracle_cache_append(int(kind), slots, _ptr(k_cache), _ptr(v_cache),
                                      int(pos0), n, _ptr(kn), _ptr(vn))
    if rc != 0:
        raise ValueError(f"mg_oracle_cache_append failed: {rc}")


def cache_commit(kind, k_cache, v_cache, pos0, count, k_block, v_block):
    """Speculative commit ("Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析",
    section "第三招：D-Flash投机解码实现3倍提速": the main model checks a drafted
    block in one pass and keeps what it accepts).  The kept tokens are the first
    `count` of the block; the cache must then hold the linear history of kept
    tokens only, which is the append of that prefix and nothing else."""
    if not 0 <= count <= len(k_block):
        raise ValueError(f"commit count {count} outside [0, {len(k_block)}]")
    if count:
        cache_append(kind, k_cache, v_cache, pos0, k_block[:count], v_block[:count])


def paged_append(k_pool, v_pool, table_row, page_size, pos0, k_new, v_new):
    """Paged global cache ("Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳
    Muse Glimmer", "窄缓存为长上下文留出空间": page size and fragmentation set
    the memory actually used).  Position p of the sequence is row p % page_size
    of page table_row[p // page_size] of the pool ([num_pages][2][page_size][128]
    uint16 bit patterns, in place)."""
    kn = bits(k_new)
    vn = bits(v_new)
    for t in range(kn.shape[0]):
        p = pos0 + t
        page = int(table_row[p // page_size])
        if not 0 <= page < k_pool.shape[0]:
            raise ValueError(f"position {p}: page {page} outside the pool")
        k_pool[page, :, p % page_size, :] = kn[t]
        v_pool[page, :, p % page_size, :] = vn[t]


def paged_history(k_pool, v_pool, table_row, page_size, upto):
    """Rows 0 .. upto-1 of a sequence read back through its page table, as a
    linear history ([upto][2][128] uint16, the layout attention() takes)."""
    k = np.empty((upto, 2, D), np.uint16)
    v = np.empty((upto, 2, D), np.uint16)
    for p in range(upto):
        page = int(table_row[p // page_size])
        k[p] = k_pool[page, :, p % page_size, :]
        v[p] = v_pool[page, :, p % page_size, :]
    return k, v


# ----------------------------------------------------------- FP8 cache ----
# An FP8 KV cache for global layers: e4m3 codes with one power-of-two scale
# per KV head for K and one for V (the pages list cache quantisation as a way
# to shrink the cache, "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳
# Muse Glimmer", "窄缓存为长上下文留出空间").  e4m3 here is the OCP FP8 E4M3
# format: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
# holds the subnormals m * 2^-9; no infinities; S.1111.111 is NaN, so the
# largest finite magnitude is 1.75 * 2^8 = 448.

E4M3_MAX = 448.0

# Column of a position inside its 16-position group of a transposed V tile:
# positions 2t, 2t+1 go to columns 4t, 4t+1 and positions 8+2t, 9+2t to
# columns 4t+2, 4t+3 (t = 0..3).
E4M3_V_COLUMN = [4 * ((j % 8) // 2) + 2 * (j // 8) + (j % 2) for j in range(16)]


def e4m3_encode(x):
    """float64 array -> uint8 e4m3 codes: round to nearest, ties to even,
    magnitudes above 448 saturate to 448, the sign of zero is kept."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(a)                           # a = f * 2^ex, f in [0.5, 1)
    binade = np.maximum(ex - 1, -6)               # below 2^-6 the spacing stays 2^-9
    quantum = np.ldexp(1.0, binade - 3)           # 3 mantissa bits
    r = a / quantum                               # exact: power-of-two divisor
    n = np.floor(r)
    frac = r - n
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(n, 2.0) == 1.0))
    v = np.minimum((n + up) * quantum, E4M3_MAX)  # a carry may move up one binade
    _, ev = np.frexp(v)
    e_field = np.where(v >= 2.0 ** -6, ev - 1 + 7, 0)
    mant = np.where(e_field == 0, v / 2.0 ** -9, (np.ldexp(v, -(e_field - 7)) - 1.0) * 8.0)
    code = (e_field * 8 + mant).astype(np.int64) | (neg.astype(np.int64) << 7)
    return code.astype(np.uint8)


def e4m3_decode(code):
    """uint8 e4m3 codes -> float64 values (NaN for the NaN codes)."""
    c = np.asarray(code).astype(np.int64)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where((c >> 7) & 1 == 1, -v, v)


def _check_pow2(scales):
    for s in scales:
        m, _ = np.frexp(float(s))
        if not (s > 0 and m == 0.5):
            raise ValueError(f"scale {s} is not a positive power of two")


def _e4m3_v_columns(pos):
    """Column of each position inside its transposed 64-position V tile."""
    pos = np.asarray(pos)
    return 16 * ((pos % 64) // 16) + np.asarray(E4M3_V_COLUMN)[pos % 16]


def e4m3_cache_append(k_codes, vt_codes, k_scale, v_scale, pos0, k_new, v_new):
    """Store positions pos0 .. pos0+n-1 of one sequence in an FP8 cache (in
    place).  K: k_codes[g][p][d] = e4m3(k / k_scale[g]).  V, transposed per
    64-position tile: vt_codes[g][p // 64][d][16 * ((p % 64) // 16) +
    E4M3_V_COLUMN[p % 16]] = e4m3(v / v_scale[g]).  Scales are powers of two,
    so the division is exact and the code is the value's correct rounding."""
    _check_pow2(list(k_scale) + list(v_scale))
    kf = (bits(k_new).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    vf = (bits(v_new).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    n = kf.shape[0]
    pos = np.arange(pos0, pos0 + n)
    tiles, cols = pos // 64, _e4m3_v_columns(pos)
    dims = np.arange(D)
    for g in range(HKV):
        k_codes[g, pos0:pos0 + n, :] = e4m3_encode(kf[:, g, :] / k_scale[g])
        vt_codes[g, tiles[:, None], dims[None, :], cols[:, None]] = e4m3_encode(vf[:, g, :] / v_scale[g])


def e4m3_history(k_codes, vt_codes, k_scale, v_scale, upto):
    """Positions 0 .. upto-1 of an FP8 cache dequantised (code value x scale,
    exactly representable in bf16), as bf16 bit patterns [upto][2][128] for
    attention()."""
    pos = np.arange(upto)
    tiles, cols = pos // 64, _e4m3_v_columns(pos)
    dims = np.arange(D)
    k = np.empty((upto, HKV, D), np.float64)
    v = np.empty((upto, HKV, D), np.float64)
    for g in range(HKV):
        k[:, g, :] = e4m3_decode(k_codes[g, :upto, :]) * k_scale[g]
        v[:, g, :] = e4m3_decode(vt_codes[g, tiles[:, None], dims[None, :], cols[:, None]]) * v_scale[g]

    def to_bf16_bits(a):
        f = a.astype(np.float32)
        assert np.array_equal(f.astype(np.float64), a), "value not exact in fp32"
        b = f.view(np.uint32)
        assert not np.any(b & 0xFFFF), "value not exact in bf16"
        return (b >> 16).astype(np.uint16)
    return to_bf16_bits(k), to_bf16_bits(v)


def decode_from_cache(lay, k_cache, v_cache, p, q):
    kc = bits(k_cache); vc = bits(v_cache); qq = bits(q)
    slots = kc.shape[1]
    o = np.zeros((HQ, D), dtype=np.float64)
    rc = lib().mg_oracle_decode_from_cache(ctypes.byref(lay), slots, _ptr(kc), _ptr(vc),
                                           int(p), _ptr(qq), _ptr(o))
    if rc != 0:
        raise ValueError(f"mg_oracle_decode_from_cache failed: {rc}")
    return o


def rope(x, t, theta=THETA):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).copy())
    assert a.shape == (D,)
    lib().mg_oracle_rope(_ptr(a), float(t), float(theta))
    return a


# ------------------------------------------------------ QKV projection ----
# The step before the attention path: each token's hidden state (hidden size
# 6656; "深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？", section 01,
# which also gives the 32 query heads and 2 KV heads of dimension 128) is
# projected to its query, key and value.  Reading (the pages give only the
# sizes): one weight matrix W of 4608 x 6656 whose output features are the
# 32 query heads (features 128 h .. 128 h + 127), then the 2 key heads
# (4096 + 128 g ..), then the 2 value heads (4352 + 128 g ..); y = x W^T.
# The projected K and V are appended to the layer's cache exactly as
# cache_append does.

HIDDEN = 6656
QKV_FEATURES = (HQ + 2 * HKV) * D  # 4608


def _widen(a):
    """bf16 bit patterns (uint16 array or bf16 tensor) -> float64, exactly."""
    b = bits(a)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def qkv_project(x, w):
    """y = x W^T in float64 for x [M][6656] and W [4608][6656] (bf16 bits);
    every product of two bf16 values is exact in float64 and the sum of 6656
    of them is within a few units of 2^-53 of the exact value."""
    xd, wd = _widen(x), _widen(w)
    assert xd.ndim == 2 and xd.shape[1] == HIDDEN, xd.shape
    assert wd.shape == (QKV_FEATURES, HIDDEN), wd.shape
    return xd @ wd.T


def qkv_split(y):
    """[M][4608] -> q [M][32][128], k [M][2][128], v [M][2][128] (views)."""
    y = np.asarray(y)
    M = y.shape[0]
    q = y[:, :HQ * D].reshape(M, HQ, D)
    k = y[:, HQ * D:(HQ + HKV) * D].reshape(M, HKV, D)
    v = y[:, (HQ + HKV) * D:].reshape(M, HKV, D)
    return q, k, v


def qkv_abs_bound(x, w):
    """|x| |W|^T in float64: with it, a sum of the 6656 products accumulated
    in fp32 in any order lies within gamma_6656 = 6656 u / (1 - 6656 u),
    u = 2^-24, times this of the exact value."""
    return np.abs(_widen(x)) @ np.abs(_widen(w)).T


FP32_GAMMA_HIDDEN = HIDDEN * 2.0 ** -24 / (1 - HIDDEN * 2.0 ** -24)
