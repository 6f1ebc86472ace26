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
