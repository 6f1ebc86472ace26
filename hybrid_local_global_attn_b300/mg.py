"""ctypes binding of libmg (the C ABI in ``include/mg.h``).

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of ``libmg.so``.  Functions keep the C names; tensors are torch
tensors on the GPU (bf16 data, int32 positions, uint32 error word), the
stream defaults to torch's current stream.  There is no CPU fallback: the
import fails if the library has not been built, and a call on a machine
without a GPU fails in the library.
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmg.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m hybrid_local_global_attn_b300.build` (nvcc, sm_103a)")
lib = ctypes.CDLL(LIB_PATH)

HQ, HKV, D = 32, 2, 128
WINDOW = 2048
VERIFY_MAX = 16
N_LAYERS = 52
LOCAL, GLOBAL = 0, 1
BF16, E4M3 = 0, 1
OP_DECODE, OP_VERIFY, OP_PREFILL = 0, 1, 2
DERR_POSITION, DERR_TIMEOUT, DERR_COUNT, DERR_PAGE = 1, 2, 4, 8
ROPE_THETA = 10000.0
SCALE = 1.0 / math.sqrt(D)


class mg_layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("scale", ctypes.c_float)]


class mg_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("slots", ctypes.c_int32),
                ("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float * 2), ("v_scale", ctypes.c_float * 2)]


_P = ctypes.c_void_p
_i32 = ctypes.c_int32
_LP = ctypes.POINTER(mg_layer)
_CP = ctypes.POINTER(mg_cache)
lib.mg_cache_bytes.argtypes = [_i32, _i32, _i32]
lib.mg_cache_bytes.restype = ctypes.c_size_t
lib.mg_e4m3_cache_bytes.argtypes = [_i32, _i32]
lib.mg_e4m3_cache_bytes.restype = ctypes.c_size_t
lib.mg_page_pool_bytes.argtypes = [_i32, _i32]
lib.mg_page_pool_bytes.restype = ctypes.c_size_t
lib.mg_workspace_bytes.argtypes = [_i32, _LP, _i32, _i32, _i32]
lib.mg_workspace_bytes.restype = ctypes.c_size_t
lib.mg_status_str.argtypes = [ctypes.c_int]
lib.mg_status_str.restype = ctypes.c_char_p
lib.mg_layer_kind.argtypes = [_i32]
lib.mg_decode_kernel_count.argtypes = [_LP, _i32, _i32]
lib.mg_decode_kernel_count.restype = ctypes.c_int
lib.mg_layer_kind.restype = ctypes.c_int
lib.mg_kv_append.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, _P]
lib.mg_kv_commit.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, _P, _P, _P]
lib.mg_kv_commit_layers.argtypes = [_i32, _LP, _CP, _P, _i32, _P, _P, _P, _P, _P, _P]
lib.mg_attn_decode.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, ctypes.c_size_t, _P, _P]
lib.mg_append_decode.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
lib.mg_append_decode_ex.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                    ctypes.c_uint32, _P]
lib.mg_attn_verify.argtypes = [_LP, _CP, _P, _i32, _i32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
lib.mg_attn_prefill.argtypes = [_LP, _CP, _P, _i32, _i32, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
lib.mg_qkv_workspace_bytes.argtypes = [_i32, _i32]
lib.mg_qkv_workspace_bytes.restype = ctypes.c_size_t
lib.mg_qkv_append.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
lib.mg_qkv_append.restype = ctypes.c_int
lib.mg_debug_decode_stall.argtypes = [_LP, _CP, _P, _i32, _P, _P, _P, ctypes.c_size_t, _P, _P,
                                      ctypes.c_uint64, _i32]
lib.mg_debug_decode_stall.restype = ctypes.c_int
for _f in (lib.mg_kv_append, lib.mg_kv_commit, lib.mg_kv_commit_layers, lib.mg_attn_decode, lib.mg_append_decode,
           lib.mg_append_decode_ex, lib.mg_attn_verify, lib.mg_attn_prefill):
    _f.restype = ctypes.c_int


class MgError(RuntimeError):
    def __init__(self, status):
        self.status = status
        super().__init__(f"libmg: {mg_status_str(status)} (status {status})")


def mg_status_str(status: int) -> str:
    return lib.mg_status_str(int(status)).decode()


def mg_cache_bytes(kind: int, batch: int, capacity: int) -> int:
    return int(lib.mg_cache_bytes(kind, batch, capacity))


def mg_e4m3_cache_bytes(batch: int, capacity: int) -> int:
    return int(lib.mg_e4m3_cache_bytes(batch, capacity))


def mg_page_pool_bytes(num_pages: int, page_size: int) -> int:
    return int(lib.mg_page_pool_bytes(num_pages, page_size))


def mg_decode_kernel_count(layer, batch: int, max_len: int) -> int:
    return int(lib.mg_decode_kernel_count(ctypes.byref(layer), batch, max_len))


def mg_layer_kind(l: int) -> int:
    return int(lib.mg_layer_kind(l))


def make_layer(kind: int, rope_theta: float = ROPE_THETA, scale: float = SCALE) -> mg_layer:
    return mg_layer(int(kind), WINDOW if kind == LOCAL else 0,
                    float(rope_theta) if kind == LOCAL else 0.0, float(scale))


def mg_workspace_bytes(op: int, layer: mg_layer, batch: int, n: int, max_len: int) -> int:
    v = int(lib.mg_workspace_bytes(op, ctypes.byref(layer), batch, n, max_len))
    if v == ctypes.c_size_t(-1).value:
        raise MgError(1)
    return v


class KVCache:
    """One layer's cache: k and v bf16 [batch][2][slots][128] on the GPU."""

    def __init__(self, kind: int, batch: int, capacity: int = 0, device="cuda"):
        self.kind = kind
        self.batch = batch
        self.slots = WINDOW if kind == LOCAL else int(capacity)
        self.k = torch.zeros((batch, HKV, self.slots, D), dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)
        self.struct = mg_cache(self.k.data_ptr(), self.v.data_ptr(), batch, self.slots)

    def nbytes(self) -> int:
        return self.k.numel() * 2 + self.v.numel() * 2


class PagedKVCache:
    """A global layer's paged cache: k and v pools bf16 [num_pages][2][page_size][128]
    shared by the batch, and a page table int32 [batch][capacity // page_size]
    (all on the GPU; the table is the caller's to fill, -1 = unassigned)."""

    def __init__(self, batch: int, capacity: int, num_pages: int, page_size: int = 256,
                 device="cuda"):
        if capacity % page_size:
            raise ValueError("capacity must be a multiple of page_size")
        self.kind = GLOBAL
        self.batch = batch
        self.slots = int(capacity)
        self.page_size = int(page_size)
        self.num_pages = int(num_pages)
        self.k = torch.zeros((num_pages, HKV, page_size, D), dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)
        self.table = torch.full((batch, capacity // page_size), -1, dtype=torch.int32, device=device)
        self.struct = mg_cache(self.k.data_ptr(), self.v.data_ptr(), batch, self.slots,
                               self.table.data_ptr(), self.page_size, self.num_pages)

    def nbytes(self) -> int:
        return self.k.numel() * 2 + self.v.numel() * 2

    def linear(self, b: int, upto: int):
        """Sequence b's rows [0, upto) gathered through the table: (k, v) [2][upto][128]."""
        ps = self.page_size
        pages = self.table[b, :(upto + ps - 1) // ps].long()
        k = self.k[pages].permute(1, 0, 2, 3).reshape(HKV, -1, D)[:, :upto]
        v = self.v[pages].permute(1, 0, 2, 3).reshape(HKV, -1, D)[:, :upto]
        return k, v


class E4M3KVCache:
    """A global layer's FP8 cache: K codes uint8 [batch][2][slots][128], V codes
    transposed per 64-position tile uint8 [batch][2][slots // 64][128][64], and
    one power-of-two scale per KV head for K and for V."""

    def __init__(self, batch: int, capacity: int, k_scale=(1.0, 1.0), v_scale=(1.0, 1.0),
                 device="cuda"):
        slots = (int(capacity) + 63) // 64 * 64
        self.kind = GLOBAL
        self.batch = batch
        self.slots = slots
        self.k = torch.zeros((batch, HKV, slots, D), dtype=torch.uint8, device=device)
        self.v = torch.zeros((batch, HKV, slots // 64, D, 64), dtype=torch.uint8, device=device)
        self.k_scale = tuple(float(x) for x in k_scale)
        self.v_scale = tuple(float(x) for x in v_scale)
        self.struct = mg_cache(self.k.data_ptr(), self.v.data_ptr(), batch, slots, None, 0, 0, E4M3,
                               (ctypes.c_float * 2)(*self.k_scale), (ctypes.c_float * 2)(*self.v_scale))

    def nbytes(self) -> int:
        return self.k.numel() + self.v.numel()


def _ptr(t, dtype=None):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous() or (dtype is not None and t.dtype != dtype):
        raise TypeError(f"expected a contiguous CUDA tensor of {dtype}, got {t.dtype} "
                        f"on {t.device} (contiguous={t.is_contiguous()})")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _call(fn, *args):
    rc = fn(*args)
    if rc != 0:
        raise MgError(rc)


def mg_kv_append(layer, cache: KVCache, pos0, k_new, v_new, err, stream=None):
    _call(lib.mg_kv_append, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos0, torch.int32),
          int(k_new.shape[1]), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
          _ptr(err, torch.int32), _stream(stream))


def mg_kv_commit(layer, cache: KVCache, pos0, count, k_new, v_new, err, pos_next=None,
                 stream=None):
    """Write the first count[b] tokens of a verified block (k_new/v_new
    [B][n][2][128]) at pos0[b]; optionally pos_next[b] = pos0[b] + count[b]."""
    _call(lib.mg_kv_commit, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos0, torch.int32),
          int(k_new.shape[1]), _ptr(count, torch.int32), _ptr(k_new, torch.bfloat16),
          _ptr(v_new, torch.bfloat16), _ptr(pos_next, torch.int32), _ptr(err, torch.int32),
          _stream(stream))


def mg_kv_commit_layers(layers, caches, pos0, count, k_new, v_new, err, pos_next=None,
                        stream=None):
    """mg_kv_commit into every cache of `caches` in one launch; k_new/v_new
    are [n_layers][B][n][2][128]."""
    L = len(layers)
    if len(caches) != L or k_new.shape[0] != L or v_new.shape != k_new.shape:
        raise ValueError("one layer, one cache and one block per layer")
    lay_arr = (mg_layer * L)(*layers)
    cache_arr = (mg_cache * L)(*[c.struct for c in caches])
    _call(lib.mg_kv_commit_layers, L, lay_arr, cache_arr, _ptr(pos0, torch.int32), int(k_new.shape[2]),
          _ptr(count, torch.int32), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
          _ptr(pos_next, torch.int32), _ptr(err, torch.int32), _stream(stream))


def mg_attn_decode(layer, cache: KVCache, pos, max_len, q, o, ws, err, stream=None):
    _call(lib.mg_attn_decode, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos, torch.int32),
          int(max_len), _ptr(q, torch.bfloat16), _ptr(o, torch.bfloat16), _ptr(ws),
          ws.numel() * ws.element_size() if ws is not None else 0, _ptr(err, torch.int32),
          _stream(stream))


HIDDEN = 6656
QKV_FEATURES = (HQ + 2 * HKV) * D


def mg_qkv_workspace_bytes(batch: int, n: int) -> int:
    v = int(lib.mg_qkv_workspace_bytes(batch, n))
    if v == ctypes.c_size_t(-1).value:
        raise MgError(1)
    return v


def qkv_workspace(batch, n, device="cuda"):
    return torch.empty(max(mg_qkv_workspace_bytes(batch, n), 256), dtype=torch.uint8, device=device)


def mg_qkv_append(layer, cache, pos0, x, w, q_out, ws, err, k_out=None, v_out=None, stream=None):
    """Project x [B][n][6656] with w [4608][6656] to q_out [B][n][32][128] and
    append the key / value rows to `cache` at pos0[b] ..; k_out / v_out
    [B][n][2][128] optionally receive them too."""
    _call(lib.mg_qkv_append, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos0, torch.int32),
          int(x.shape[1]), _ptr(x, torch.bfloat16), _ptr(w, torch.bfloat16),
          _ptr(q_out, torch.bfloat16), _ptr(k_out, torch.bfloat16), _ptr(v_out, torch.bfloat16),
          _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
          _ptr(err, torch.int32), _stream(stream))


def mg_debug_decode_stall(layer, cache: KVCache, pos, max_len, q, o, ws, err, wait_ns: int,
                          stall_tile: int, stream=None):
    """Self-test of the bounded waits: a global-layer decode whose producer
    stops at key tile `stall_tile` of every split, with pipeline waits
    limited to wait_ns; the device error word then reports DERR_TIMEOUT."""
    _call(lib.mg_debug_decode_stall, ctypes.byref(layer), ctypes.byref(cache.struct),
          _ptr(pos, torch.int32), int(max_len), _ptr(q, torch.bfloat16), _ptr(o, torch.bfloat16),
          _ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
          _ptr(err, torch.int32), _stream(stream), int(wait_ns), int(stall_tile))


def mg_append_decode(layer, cache: KVCache, pos, max_len, q, k_new, v_new, o, ws, err, stream=None):
    _call(lib.mg_append_decode, ctypes.byref(layer), ctypes.byref(cache.struct),
          _ptr(pos, torch.int32), int(max_len), _ptr(q, torch.bfloat16), _ptr(k_new, torch.bfloat16),
          _ptr(v_new, torch.bfloat16), _ptr(o, torch.bfloat16), _ptr(ws),
          ws.numel() * ws.element_size() if ws is not None else 0, _ptr(err, torch.int32),
          _stream(stream))


EARLY_START = 1  # MG_EARLY_START
OVERLAP_NEXT = 2  # MG_OVERLAP_NEXT


def mg_append_decode_ex(layer, cache: KVCache, pos, max_len, q, k_new, v_new, o, ws, err, flags,
                        stream=None):
    _call(lib.mg_append_decode_ex, ctypes.byref(layer), ctypes.byref(cache.struct),
          _ptr(pos, torch.int32), int(max_len), _ptr(q, torch.bfloat16), _ptr(k_new, torch.bfloat16),
          _ptr(v_new, torch.bfloat16), _ptr(o, torch.bfloat16), _ptr(ws),
          ws.numel() * ws.element_size() if ws is not None else 0, _ptr(err, torch.int32),
          int(flags), _stream(stream))


def mg_attn_verify(layer, cache: KVCache, pos0, max_len, q, k_new, v_new, o, ws, err, stream=None):
    _call(lib.mg_attn_verify, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos0, torch.int32),
          int(q.shape[1]), int(max_len), _ptr(q, torch.bfloat16), _ptr(k_new, torch.bfloat16),
          _ptr(v_new, torch.bfloat16), _ptr(o, torch.bfloat16), _ptr(ws),
          ws.numel() * ws.element_size() if ws is not None else 0, _ptr(err, torch.int32),
          _stream(stream))


def mg_attn_prefill(layer, cache: KVCache, pos0, max_len, q, k_new, v_new, o, ws, err, stream=None):
    _call(lib.mg_attn_prefill, ctypes.byref(layer), ctypes.byref(cache.struct), _ptr(pos0, torch.int32),
          int(q.shape[1]), int(max_len), _ptr(q, torch.bfloat16), _ptr(k_new, torch.bfloat16),
          _ptr(v_new, torch.bfloat16), _ptr(o, torch.bfloat16), _ptr(ws),
          ws.numel() * ws.element_size() if ws is not None else 0, _ptr(err, torch.int32),
          _stream(stream))


def workspace(op, layer, batch, n, max_len, device="cuda"):
    """Caller-side workspace allocation (torch) of the size libmg asks for
    (left uninitialised: nothing in it needs to start at any value)."""
    nbytes = mg_workspace_bytes(op, layer, batch, n, max_len)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def error_word(device="cuda"):
    """Device error word (int32 view of the C uint32), zeroed."""
    return torch.zeros(1, dtype=torch.int32, device=device)
