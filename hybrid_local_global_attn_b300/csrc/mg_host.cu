// mg_host.cu -- the C ABI of libmg (declared in include/mg.h): argument
// checks, workspace layout, TMA descriptors and kernel launches.
//
// The library keeps no device state and never allocates: every buffer comes
// from the caller.  Host-side rejections return a status and launch nothing.
#include <cmath>
#include <cstring>
#include <mutex>

#include "mg_internal.h"

namespace mg {
namespace {

constexpr int kNumSms = 148;  // B300

// ------------------------------------------------------ TMA descriptors ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Small cache of encoded descriptors keyed by (address, shape, box): decode
// steps re-use the same caches and buffers, and encoding is pure host work.
struct MapKey {
  const void *base;
  uint32_t rank;
  uint32_t bytes_per_elem;  // 2: bf16, 1: e4m3 codes
  uint32_t swizzle;         // bytes: 128 or 64
  uint64_t dims[4];
  uint32_t box[4];
  bool operator==(const MapKey &o) const {
    return base == o.base && rank == o.rank && bytes_per_elem == o.bytes_per_elem &&
           swizzle == o.swizzle && std::memcmp(dims, o.dims, sizeof dims) == 0 &&
           std::memcmp(box, o.box, sizeof box) == 0;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCache = 512;
MapEntry g_maps[kMapCache];
std::mutex g_map_mu;

// Dense tensor (bf16 or bytes) whose strides derive from dims; boxes land in
// shared memory with the given swizzle (128 or 64 bytes).
bool make_map(CUtensorMap *out, const void *base, uint32_t rank, const uint64_t *dims,
              const uint32_t *box, uint32_t bytes_per_elem = 2, uint32_t swizzle = 128) {
  MapKey key{};
  key.base = base;
  key.rank = rank;
  key.bytes_per_elem = bytes_per_elem;
  key.swizzle = swizzle;
  for (uint32_t i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  size_t h = reinterpret_cast<uintptr_t>(base) >> 8;
  for (uint32_t i = 0; i < rank; ++i) h = h * 1000003u ^ (dims[i] * 31u + box[i]);
  h = h * 31u + bytes_per_elem * 7u + swizzle;
  MapEntry &e = g_maps[h % kMapCache];
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (e.used && e.key == key) {
      *out = e.map;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gdim[4], gstride[3];
  cuuint32_t gbox[4], estr[4] = {1, 1, 1, 1};
  uint64_t stride = bytes_per_elem;
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    gbox[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  CUtensorMap m;
  CUresult r = fn(&m, bytes_per_elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  rank, const_cast<void *>(base), gdim, gstride, gbox, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    e.key = key;
    e.map = m;
    e.used = true;
  }
  *out = m;
  return true;
}

// KV-like tensor [outer][rows][128] read in boxes of `box_rows` x 64 dims.
bool map_rows(CUtensorMap *m, const void *base, uint64_t rows, uint64_t outer, uint32_t box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(kD), rows, outer};
  const uint32_t box[3] = {64, box_rows, 1};
  return make_map(m, base, 3, dims, box);
}

}  // namespace

cudaError_t ensure_smem_attr(const void *kernel, int bytes, int kernel_id) {
  static std::mutex mu;
  static uint64_t done[16] = {};  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || kernel_id < 0 || kernel_id >= 16) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lk(mu);
  if (done[kernel_id] & (1ull << dev)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && (kernel_id == 2 || kernel_id == 3))  // 16-CTA clusters: a non-portable size
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[kernel_id] |= 1ull << dev;
  return e;
}

namespace {

// ---------------------------------------------------------------- RoPE ----
// w_i = theta^(-2i/128) as 0.64 fixed-point turns per position, and the
// (cos, sin) of the slot steps the local kernel takes between a thread's
// keys, all from double precision.
struct RopeTables {
  uint64_t turn[64];
  float2 step[3][64];
};

RopeTables rope_tables(float theta) {
  static std::mutex mu;
  static float last_theta = -1.f;
  static RopeTables last;
  std::lock_guard<std::mutex> lk(mu);
  if (theta != last_theta) {
    for (int i = 0; i < 64; ++i) {
      const double w = std::pow(static_cast<double>(theta), -2.0 * i / 128.0);
      const double t = w / (2.0 * M_PI);  // turns per position, < 1
      last.turn[i] = static_cast<uint64_t>(std::ldexp(t, 64));
      for (int k = 0; k < 3; ++k) {
        const double a = static_cast<double>(kRopeSteps[k]) * w;
        last.step[k][i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
      }
    }
    last_theta = theta;
  }
  return last;
}

RopeTurns rope_turns(float theta) {
  const RopeTables t = rope_tables(theta);
  RopeTurns r;
  std::memcpy(r.turn, t.turn, sizeof r.turn);
  return r;
}

// ---------------------------------------------------------- validation ----
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layer(const mg_layer *L) {
  if (L == nullptr) return MG_ERR_INVALID;
  if (L->kind != MG_LOCAL && L->kind != MG_GLOBAL) return MG_ERR_INVALID;
  if (!(L->scale > 0.f) || !std::isfinite(L->scale)) return MG_ERR_UNSUPPORTED;
  if (L->kind == MG_LOCAL) {
    if (L->window != kWindow) return MG_ERR_UNSUPPORTED;
    if (!(L->rope_theta > 1.f) || !std::isfinite(L->rope_theta)) return MG_ERR_UNSUPPORTED;
  } else if (L->window != 0) {
    return MG_ERR_UNSUPPORTED;
  }
  return MG_OK;
}

// A positive power of two whose reciprocal is also a normal float.
bool pow2_scale(float s) {
  if (!(s > 0.f) || !std::isfinite(s)) return false;
  int e = 0;
  const float m = std::frexp(s, &e);
  return m == 0.5f && e - 1 >= -126 && e - 1 <= 126;
}

int check_cache(const mg_layer *L, const mg_cache *C) {
  if (C == nullptr || C->k == nullptr || C->v == nullptr) return MG_ERR_INVALID;
  if (C->batch < 1 || C->slots < 1) return MG_ERR_INVALID;
  if (L->kind == MG_LOCAL && C->slots != kWindow) return MG_ERR_UNSUPPORTED;
  if (!aligned16(C->k) || !aligned16(C->v)) return MG_ERR_INVALID;
  if (C->dtype != MG_BF16) {
    // FP8: global layers, linear layout, whole 64-position tiles, power-of-two scales
    if (C->dtype != MG_E4M3 || L->kind != MG_GLOBAL || C->page_table != nullptr)
      return MG_ERR_UNSUPPORTED;
    if (C->slots % 64 != 0) return MG_ERR_INVALID;
    for (int g = 0; g < kHkv; ++g)
      if (!pow2_scale(C->k_scale[g]) || !pow2_scale(C->v_scale[g])) return MG_ERR_INVALID;
  }
  if (C->page_table != nullptr) {
    if (L->kind != MG_GLOBAL) return MG_ERR_UNSUPPORTED;  // the ring is never paged
    if (C->page_size < kTcKeys || C->page_size % kTcKeys != 0) return MG_ERR_UNSUPPORTED;
    if (C->slots % C->page_size != 0 || C->num_pages < 1) return MG_ERR_INVALID;
    if (static_cast<int64_t>(C->num_pages) * kHkv > 0x7fffffff) return MG_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(C->page_table) % 4 != 0) return MG_ERR_INVALID;
  }
  return MG_OK;
}

// Element type of a checked cache and, for FP8, the exact reciprocals of its
// power-of-two scales.
void set_dtype(const mg_cache *C, int32_t *dtype, float *k_mul, float *v_mul) {
  *dtype = C->dtype;
  for (int g = 0; g < kHkv; ++g) {
    k_mul[g] = C->dtype == MG_E4M3 ? 1.0f / C->k_scale[g] : 1.0f;
    v_mul[g] = C->dtype == MG_E4M3 ? 1.0f / C->v_scale[g] : 1.0f;
  }
}

// Rows of a checked cache as the kernels address them.
CacheMap cache_map(const mg_cache *C) {
  CacheMap m;
  const bool paged = C->page_table != nullptr;
  m.table = C->page_table;
  m.rows = paged ? C->page_size : C->slots;
  m.pages_per_seq = paged ? C->slots / C->page_size : 0;
  m.num_pages = paged ? C->num_pages : 0;
  return m;
}

// 3D tensor map (128 dims, rows, outer) over a checked cache's K or V.
bool map_cache(CUtensorMap *m, const mg_cache *C, const void *base, uint32_t box_rows) {
  if (C->page_table != nullptr)
    return map_rows(m, base, C->page_size, static_cast<uint64_t>(C->num_pages) * kHkv, box_rows);
  return map_rows(m, base, C->slots, static_cast<uint64_t>(C->batch) * kHkv, box_rows);
}

int splits_decode(int32_t kind, int32_t batch, int32_t max_len) {
  const int64_t n_slots = kind == MG_LOCAL ? std::min<int64_t>(max_len, kWindow) : max_len;
  const int64_t tiles = (n_slots + kDecTile - 1) / kDecTile;
  int64_t s = (2 * kNumSms) / (static_cast<int64_t>(batch) * kHkv);
  s = std::max<int64_t>(1, std::min<int64_t>(s, tiles));
  return static_cast<int>(std::min<int64_t>(s, kDecMaxSplits));
}

int splits_verify(int32_t kind, int32_t batch, int32_t n, int32_t max_len) {
  const int64_t keys = kind == MG_LOCAL ? std::min<int64_t>(max_len, kWindow) : max_len;
  const int64_t tiles = (keys + kTcKeys - 1) / kTcKeys;
  const int64_t qblocks = (n + kTcPosPerCta - 1) / kTcPosPerCta;
  int64_t s = kNumSms / (static_cast<int64_t>(batch) * kHkv * qblocks);
  s = std::max<int64_t>(1, std::min<int64_t>(s, tiles));
  return static_cast<int>(std::min<int64_t>(s, kTcMaxSplits));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t part_o, part_lse, qs, qs_lo, ks, ks_lo, vs, total;
  int splits, R;
};

// Returns false for arguments no layout exists for.
bool ws_layout(int32_t op, const mg_layer *L, int32_t batch, int32_t n, int32_t max_len,
               WsLayout *w) {
  std::memset(w, 0, sizeof *w);
  if (L == nullptr || batch < 1 || n < 1 || max_len < 1) return false;
  size_t off = 0;
  const bool local = L->kind == MG_LOCAL;
  if (op == MG_OP_DECODE) {
    if (n != 1) return false;
    if (local) {
      // one cluster per (sequence, KV head) merges in shared memory: no workspace
      w->splits = kLocCluster;
    } else {
      // one split: the kernel writes o directly and needs no workspace
      w->splits = splits_decode(L->kind, batch, max_len);
      if (w->splits > 1) {
        const size_t rows = static_cast<size_t>(batch) * kHq;
        w->part_o = off;
        off = align256(off + rows * w->splits * kD * sizeof(float));
        w->part_lse = off;
        off = align256(off + rows * w->splits * sizeof(float));
      }
    }
  } else if (op == MG_OP_VERIFY && local) {
    // the ring kernels: one cluster per (sequence, KV head) for one token (no
    // workspace); for a block, one per (sequence, KV head, 8 tokens), whose
    // CTAs exchange their partial rows through the workspace
    if (n > MG_VERIFY_MAX) return false;
    w->splits = kLocCluster;
    if (n > 1) {
      const int64_t triples =
          static_cast<int64_t>(batch) * kHkv * ((n + kTcPosPerTile - 1) / kTcPosPerTile);
      const size_t slots = static_cast<size_t>(triples) * kGroup * local_tc_cluster(triples) * kTcPosPerTile;
      w->part_o = off;
      off = align256(off + slots * kD * sizeof(float));
      w->part_lse = off;
      off = align256(off + slots * sizeof(float));
    }
  } else if (op == MG_OP_VERIFY || op == MG_OP_PREFILL) {
    if (op == MG_OP_VERIFY && n > MG_VERIFY_MAX) return false;
    w->splits = op == MG_OP_VERIFY ? splits_verify(L->kind, batch, n, max_len) : 1;
    if (w->splits > 1) {
      const size_t rows = static_cast<size_t>(batch) * n * kHq;
      w->part_o = off;
      off = align256(off + rows * w->splits * kD * sizeof(float));
      w->part_lse = off;
      off = align256(off + rows * w->splits * sizeof(float));
    }
    if (local) {  // staged operands: rotated q and k as bf16 hi and lo halves, and v
      w->R = kWindow + n;
      w->qs = off;
      off = align256(off + static_cast<size_t>(batch) * n * kHq * kD * 2);
      w->qs_lo = off;
      off = align256(off + static_cast<size_t>(batch) * n * kHq * kD * 2);
      w->ks = off;
      off = align256(off + static_cast<size_t>(batch) * kHkv * w->R * kD * 2);
      w->ks_lo = off;
      off = align256(off + static_cast<size_t>(batch) * kHkv * w->R * kD * 2);
      w->vs = off;
      off = align256(off + static_cast<size_t>(batch) * kHkv * w->R * kD * 2);
    }
  } else {
    return false;
  }
  w->total = off;
  return true;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? MG_OK : MG_ERR_CUDA; }


template <typename T>
T *at(void *base, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(base) + off);
}

// Local layers, decode and verify: the ring kernel, n query tokens per
// sequence starting at d_pos; block rows (k_new, v_new) optional.
cudaError_t launch_local(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                         int32_t n, int32_t max_len, const void *q, const void *k_new,
                         const void *v_new, bool write_new, void *o, uint32_t *d_err,
                         const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t s,
                         bool early = false, float *x_rows = nullptr, float *x_lse = nullptr,
                         bool overlap = false) {
  LocalParams p;
  p.pos = d_pos;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.err = d_err;
  p.batch = cache->batch;
  p.n = n;
  p.max_len = max_len;
  p.write_new = write_new ? 1 : 0;
  p.early = early ? 1 : 0;
  p.overlap = overlap ? 1 : 0;
  p.x_rows = x_rows;
  p.x_lse = x_lse;
  p.scale_log2 = layer->scale * static_cast<float>(M_LOG2E);
  const RopeTables t = rope_tables(layer->rope_theta);
  std::memcpy(p.turn, t.turn, sizeof p.turn);
  std::memcpy(p.step, t.step, sizeof p.step);
  return n > 1 ? launch_local_tc(p, tk, tv, s) : launch_local_attn(p, tk, tv, s);
}

}  // namespace
}  // namespace mg

using namespace mg;

extern "C" {

size_t mg_cache_bytes(int32_t kind, int32_t batch, int32_t capacity) {
  if (batch < 0) return 0;
  int64_t slots;
  if (kind == MG_LOCAL) slots = kWindow;
  else if (kind == MG_GLOBAL) {
    if (capacity < 0) return 0;
    slots = capacity;
  } else return 0;
  return static_cast<size_t>(2) * batch * kHkv * slots * kD * 2;
}

size_t mg_e4m3_cache_bytes(int32_t batch, int32_t capacity) {
  if (batch < 0 || capacity < 0 || capacity % 64 != 0) return 0;
  return static_cast<size_t>(2) * batch * kHkv * capacity * kD;
}

size_t mg_page_pool_bytes(int32_t num_pages, int32_t page_size) {
  if (num_pages < 0 || page_size < kTcKeys || page_size % kTcKeys != 0) return 0;
  return static_cast<size_t>(2) * num_pages * kHkv * page_size * kD * 2;
}

size_t mg_workspace_bytes(int32_t op, const mg_layer *layer, int32_t batch, int32_t n,
                          int32_t max_len) {
  if (check_layer(layer) != MG_OK) return static_cast<size_t>(-1);
  WsLayout w;
  if (!ws_layout(op, layer, batch, n, max_len, &w)) return static_cast<size_t>(-1);
  return w.total;
}

int mg_decode_kernel_count(const mg_layer *layer, int32_t batch, int32_t max_len) {
  if (check_layer(layer) != MG_OK) return -1;
  WsLayout w;
  if (!ws_layout(MG_OP_DECODE, layer, batch, 1, max_len, &w)) return -1;
  return (layer->kind == MG_LOCAL || w.splits == 1) ? 1 : 2;
}

const char *mg_status_str(int status) {
  switch (status) {
    case MG_OK: return "ok";
    case MG_ERR_INVALID: return "invalid argument";
    case MG_ERR_UNSUPPORTED: return "unsupported shape or layer parameters";
    case MG_ERR_CAPACITY: return "max_len beyond the cache capacity";
    case MG_ERR_WORKSPACE: return "workspace too small";
    case MG_ERR_CUDA: return "CUDA launch or driver call failed";
    default: return "unknown status";
  }
}

int mg_layer_kind(int32_t l) {
  if (l < 0 || l >= 52) return -1;
  return (l % 4 == 3) ? MG_GLOBAL : MG_LOCAL;
}

int mg_kv_append(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0, int32_t n,
                 const void *k_new, const void *v_new, uint32_t *d_err, void *stream) {
  int st = check_layer(layer);
  if (st != MG_OK) return st;
  if ((st = check_cache(layer, cache)) != MG_OK) return st;
  if (n < 0 || d_pos0 == nullptr || d_err == nullptr) return MG_ERR_INVALID;
  if (n == 0) return MG_OK;
  if (k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new))
    return MG_ERR_INVALID;
  AppendParams p;
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
  p.pos0 = d_pos0;
  p.count = nullptr;
  p.pos_next = nullptr;
  p.err = d_err;
  p.batch = cache->batch;
  p.n = n;
  p.slots = cache->slots;
  p.kind = layer->kind;
  p.map = cache_map(cache);
  set_dtype(cache, &p.dtype, p.k_mul, p.v_mul);
  return launch_status(launch_kv_append(p, static_cast<cudaStream_t>(stream)));
}

int mg_kv_commit(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0, int32_t n,
                 const int32_t *d_count, const void *k_new, const void *v_new,
                 int32_t *d_pos_next, uint32_t *d_err, void *stream) {
  int st = check_layer(layer);
  if (st != MG_OK) return st;
  if ((st = check_cache(layer, cache)) != MG_OK) return st;
  if (n < 0 || d_pos0 == nullptr || d_count == nullptr || d_err == nullptr) return MG_ERR_INVALID;
  if (d_pos_next != nullptr && static_cast<const void *>(d_pos_next) == static_cast<const void *>(d_pos0))
    return MG_ERR_INVALID;
  if (n == 0) return MG_OK;
  if (k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new))
    return MG_ERR_INVALID;
  AppendParams p;
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
  p.pos0 = d_pos0;
  p.count = d_count;
  p.pos_next = d_pos_next;
  p.err = d_err;
  p.batch = cache->batch;
  p.n = n;
  p.slots = cache->slots;
  p.kind = layer->kind;
  p.map = cache_map(cache);
  set_dtype(cache, &p.dtype, p.k_mul, p.v_mul);
  return launch_status(launch_kv_append(p, static_cast<cudaStream_t>(stream)));
}

int mg_kv_commit_layers(int32_t n_layers, const mg_layer *layers, const mg_cache *caches,
                        const int32_t *d_pos0, int32_t n, const int32_t *d_count,
                        const void *k_new, const void *v_new, int32_t *d_pos_next,
                        uint32_t *d_err, void *stream) {
  if (n_layers < 1 || n_layers > MG_COMMIT_MAX_LAYERS || layers == nullptr || caches == nullptr)
    return MG_ERR_INVALID;
  for (int32_t l = 0; l < n_layers; ++l) {
    int st = check_layer(&layers[l]);
    if (st != MG_OK) return st;
    if ((st = check_cache(&layers[l], &caches[l])) != MG_OK) return st;
    if (caches[l].batch != caches[0].batch) return MG_ERR_INVALID;
  }
  if (n < 0 || d_pos0 == nullptr || d_count == nullptr || d_err == nullptr) return MG_ERR_INVALID;
  if (d_pos_next != nullptr && static_cast<const void *>(d_pos_next) == static_cast<const void *>(d_pos0))
    return MG_ERR_INVALID;
  if (n == 0) return MG_OK;
  if (k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new))
    return MG_ERR_INVALID;
  CommitLayersParams p;
  std::memset(&p, 0, sizeof p);
  p.common.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.common.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.common.pos0 = d_pos0;
  p.common.count = d_count;
  p.common.pos_next = d_pos_next;
  p.common.err = d_err;
  p.common.batch = caches[0].batch;
  p.common.n = n;
  for (int32_t l = 0; l < n_layers; ++l) {
    p.k_cache[l] = static_cast<__nv_bfloat16 *>(caches[l].k);
    p.v_cache[l] = static_cast<__nv_bfloat16 *>(caches[l].v);
    p.slots[l] = caches[l].slots;
    p.kind[l] = layers[l].kind;
    p.map[l] = cache_map(&caches[l]);
    set_dtype(&caches[l], &p.dtype[l], p.k_mul[l], p.v_mul[l]);
  }
  p.layer_stride = static_cast<size_t>(caches[0].batch) * n * kHkv * kD;
  p.layers = n_layers;
  return launch_status(launch_kv_commit_layers(p, static_cast<cudaStream_t>(stream)));
}

static int decode_impl(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                       int32_t max_len, const void *q, const void *k_new, const void *v_new,
                       void *o, void *ws, size_t ws_bytes, uint32_t *d_err, void *stream,
                       uint64_t wait_ns = kWaitLimitNs, int32_t stall_tile = -1,
                       bool early = false, bool overlap = false) {
  int st = check_layer(layer);
  if (st != MG_OK) return st;
  if ((st = check_cache(layer, cache)) != MG_OK) return st;
  if (d_pos == nullptr || d_err == nullptr || q == nullptr || o == nullptr) return MG_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o)) return MG_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return MG_ERR_INVALID;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return MG_ERR_INVALID;
  if (max_len < 1) return MG_ERR_INVALID;
  if (layer->kind == MG_GLOBAL && max_len > cache->slots) return MG_ERR_CAPACITY;
  WsLayout w;
  if (!ws_layout(MG_OP_DECODE, layer, cache->batch, 1, max_len, &w)) return MG_ERR_INVALID;
  if (ws_bytes < w.total || (w.total > 0 && ws == nullptr)) return MG_ERR_WORKSPACE;
  if (w.total > 0 && !aligned16(ws)) return MG_ERR_INVALID;
  CUtensorMap tk, tv;
  const bool e4m3 = cache->dtype == MG_E4M3;
  if (e4m3) {
    // K codes: (128 bytes, slots, batch x heads); V codes: transposed tiles
    // (64 positions, 128 dims, slots / 64, batch x heads)
    const uint64_t outer = static_cast<uint64_t>(cache->batch) * kHkv;
    const uint64_t kd[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(cache->slots), outer};
    const uint32_t kb[3] = {static_cast<uint32_t>(kD), kE4m3Tile, 1};
    const uint64_t vd[4] = {64, static_cast<uint64_t>(kD), static_cast<uint64_t>(cache->slots / 64),
                            outer};
    const uint32_t vb[4] = {64, static_cast<uint32_t>(kD), kE4m3Tile / 64, 1};
    if (!make_map(&tk, cache->k, 3, kd, kb, 1, 128) || !make_map(&tv, cache->v, 4, vd, vb, 1, 64))
      return MG_ERR_CUDA;
  } else if (!map_cache(&tk, cache, cache->k, kDecTile) ||
             !map_cache(&tv, cache, cache->v, kDecTile)) {
    return MG_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (layer->kind == MG_LOCAL)
    return launch_status(launch_local(layer, cache, d_pos, 1, max_len, q, k_new, v_new,
                                      k_new != nullptr, o, d_err, tk, tv, s, early, nullptr,
                                      nullptr, overlap));
  DecodeParams p;
  p.pos = d_pos;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
  const bool split = w.splits > 1;
  p.part_o = split ? at<float>(ws, w.part_o) : nullptr;
  p.part_lse = split ? at<float>(ws, w.part_lse) : nullptr;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.err = d_err;
  p.batch = cache->batch;
  p.slots = cache->slots;
  p.splits = w.splits;
  p.max_len = max_len;
  p.scale_log2 = layer->scale * static_cast<float>(M_LOG2E);
  p.map = cache_map(cache);
  for (int g = 0; g < kHkv; ++g) {
    p.k_scale[g] = e4m3 ? cache->k_scale[g] : 1.0f;
    p.v_scale[g] = e4m3 ? cache->v_scale[g] : 1.0f;
  }
  p.wait_ns = wait_ns;
  p.stall_tile = stall_tile;
  p.early = early && !e4m3 ? 1 : 0;
  p.overlap = overlap && p.map.table == nullptr ? 1 : 0;
  cudaError_t e = e4m3 ? launch_decode_e4m3(p, tk, tv, s) : launch_decode(p, tk, tv, s);
  if (e != cudaSuccess) return MG_ERR_CUDA;
  if (!split) return MG_OK;
  CombineParams c;
  c.part_o = p.part_o;
  c.part_lse = p.part_lse;
  c.o = static_cast<__nv_bfloat16 *>(o);
  c.rows = cache->batch * kHq;
  c.splits = w.splits;
  c.overlap = p.overlap;
  return launch_status(launch_combine(c, s));
}

int mg_attn_decode(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                   int32_t max_len, const void *q, void *o, void *ws, size_t ws_bytes,
                   uint32_t *d_err, void *stream) {
  return decode_impl(layer, cache, d_pos, max_len, q, nullptr, nullptr, o, ws, ws_bytes, d_err,
                     stream);
}

size_t mg_qkv_workspace_bytes(int32_t batch, int32_t n) {
  if (batch < 1 || n < 1) return static_cast<size_t>(-1);
  const int64_t M = static_cast<int64_t>(batch) * n;
  if (M > 0x7fffffff / kQkvFeatures) return static_cast<size_t>(-1);
  const int splits = qkv_splits(static_cast<int32_t>(M));
  return splits > 1 ? align256(static_cast<size_t>(splits) * M * kQkvFeatures * sizeof(float)) : 0;
}

int mg_qkv_append(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0, int32_t n,
                  const void *x, const void *w, void *q_out, void *k_out, void *v_out, void *ws,
                  size_t ws_bytes, uint32_t *d_err, void *stream) {
  int st = check_layer(layer);
  if (st != MG_OK) return st;
  if ((st = check_cache(layer, cache)) != MG_OK) return st;
  if (cache->dtype != MG_BF16) return MG_ERR_UNSUPPORTED;
  if (d_pos0 == nullptr || d_err == nullptr || x == nullptr || w == nullptr || q_out == nullptr)
    return MG_ERR_INVALID;
  if ((k_out == nullptr) != (v_out == nullptr)) return MG_ERR_INVALID;
  if (!aligned16(x) || !aligned16(w) || !aligned16(q_out) ||
      (k_out != nullptr && (!aligned16(k_out) || !aligned16(v_out))))
    return MG_ERR_INVALID;
  if (n < 1) return MG_ERR_INVALID;
  const size_t need = mg_qkv_workspace_bytes(cache->batch, n);
  if (need == static_cast<size_t>(-1)) return MG_ERR_INVALID;
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return MG_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return MG_ERR_INVALID;
  const int32_t M = cache->batch * n;
  CUtensorMap tx, tw;
  {
    const uint64_t xd[2] = {static_cast<uint64_t>(kHidden), static_cast<uint64_t>(M)};
    const uint32_t xb[2] = {64, 128};
    const uint64_t wd[2] = {static_cast<uint64_t>(kHidden), static_cast<uint64_t>(kQkvFeatures)};
    const uint32_t wb[2] = {64, 256};
    if (!make_map(&tx, x, 2, xd, xb) || !make_map(&tw, w, 2, wd, wb)) return MG_ERR_CUDA;
  }
  QkvParams p;
  std::memset(&p, 0, sizeof p);
  p.pos0 = d_pos0;
  p.q_out = static_cast<__nv_bfloat16 *>(q_out);
  p.k_out = static_cast<__nv_bfloat16 *>(k_out);
  p.v_out = static_cast<__nv_bfloat16 *>(v_out);
  p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
  p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
  p.part = static_cast<float *>(ws);
  p.err = d_err;
  p.M = M;
  p.n = n;
  p.batch = cache->batch;
  p.kind = layer->kind;
  p.slots = cache->slots;
  p.splits = qkv_splits(M);
  p.map = cache_map(cache);
  return launch_status(launch_qkv(p, tx, tw, static_cast<cudaStream_t>(stream)));
}

int mg_debug_decode_stall(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                          int32_t max_len, const void *q, void *o, void *ws, size_t ws_bytes,
                          uint32_t *d_err, void *stream, uint64_t wait_ns, int32_t stall_tile) {
  if (layer == nullptr || cache == nullptr) return MG_ERR_INVALID;
  if (layer->kind != MG_GLOBAL || cache->dtype != MG_BF16) return MG_ERR_UNSUPPORTED;
  if (stall_tile < 0 || wait_ns == 0 || wait_ns > kWaitLimitNs) return MG_ERR_INVALID;
  return decode_impl(layer, cache, d_pos, max_len, q, nullptr, nullptr, o, ws, ws_bytes, d_err,
                     stream, wait_ns, stall_tile);
}

int mg_append_decode(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                     int32_t max_len, const void *q, const void *k_new, const void *v_new, void *o,
                     void *ws, size_t ws_bytes, uint32_t *d_err, void *stream) {
  if (k_new == nullptr || v_new == nullptr) return MG_ERR_INVALID;
  return decode_impl(layer, cache, d_pos, max_len, q, k_new, v_new, o, ws, ws_bytes, d_err,
                     stream);
}

int mg_append_decode_ex(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos,
                        int32_t max_len, const void *q, const void *k_new, const void *v_new,
                        void *o, void *ws, size_t ws_bytes, uint32_t *d_err, uint32_t flags,
                        void *stream) {
  if (k_new == nullptr || v_new == nullptr) return MG_ERR_INVALID;
  if ((flags & ~(MG_EARLY_START | MG_OVERLAP_NEXT)) != 0) return MG_ERR_INVALID;
  return decode_impl(layer, cache, d_pos, max_len, q, k_new, v_new, o, ws, ws_bytes, d_err,
                     stream, kWaitLimitNs, -1, (flags & MG_EARLY_START) != 0,
                     (flags & MG_OVERLAP_NEXT) != 0);
}

}  // extern "C"

namespace mg {
namespace {

// Shared body of verify and prefill.
int block_attention(int32_t op, const mg_layer *layer, const mg_cache *cache,
                    const int32_t *d_pos0, int32_t n, int32_t max_len, const void *q,
                    const void *k_new, const void *v_new, void *o, void *ws, size_t ws_bytes,
                    uint32_t *d_err, cudaStream_t s) {
  int st = check_layer(layer);
  if (st != MG_OK) return st;
  if ((st = check_cache(layer, cache)) != MG_OK) return st;
  if (d_pos0 == nullptr || d_err == nullptr || q == nullptr || o == nullptr ||
      k_new == nullptr || v_new == nullptr)
    return MG_ERR_INVALID;
  if (cache->dtype != MG_BF16) return MG_ERR_UNSUPPORTED;  // FP8 caches: decode only
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_new) || !aligned16(v_new))
    return MG_ERR_INVALID;
  if (n < 1) return MG_ERR_INVALID;
  if (op == MG_OP_VERIFY && n > MG_VERIFY_MAX) return MG_ERR_UNSUPPORTED;
  if (max_len < n) return MG_ERR_INVALID;
  // the cache must hold every position before the block
  if (layer->kind == MG_GLOBAL && static_cast<int64_t>(max_len) - n > cache->slots)
    return MG_ERR_CAPACITY;
  WsLayout w;
  if (!ws_layout(op, layer, cache->batch, n, max_len, &w)) return MG_ERR_INVALID;
  if (ws_bytes < w.total || (w.total > 0 && ws == nullptr)) return MG_ERR_WORKSPACE;
  if (w.total > 0 && !aligned16(ws)) return MG_ERR_INVALID;
  const int32_t B = cache->batch;
  const bool local = layer->kind == MG_LOCAL;
  const uint64_t outer = static_cast<uint64_t>(B) * kHkv;

  if (local && op == MG_OP_VERIFY) {
    // one token: the mma.sync ring kernel; a block: the tcgen05 ring kernel
    const uint32_t rows = n == 1 ? kDecTile : kWindow / kLocCluster;
    CUtensorMap tk, tv;
    if (!map_rows(&tk, cache->k, cache->slots, outer, rows) ||
        !map_rows(&tv, cache->v, cache->slots, outer, rows))
      return MG_ERR_CUDA;
    return launch_status(launch_local(layer, cache, d_pos0, n, max_len, q, k_new, v_new, false, o,
                                      d_err, tk, tv, s, false,
                                      n > 1 ? at<float>(ws, w.part_o) : nullptr,
                                      n > 1 ? at<float>(ws, w.part_lse) : nullptr));
  }
  const void *qsrc = q;
  CUtensorMap tq, tka, tva, tkb, tvb, tql, tkl;
  if (local) {
    StageParams sp;
    sp.pos0 = d_pos0;
    sp.q = static_cast<const __nv_bfloat16 *>(q);
    sp.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    sp.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    sp.k_cache = static_cast<const __nv_bfloat16 *>(cache->k);
    sp.v_cache = static_cast<const __nv_bfloat16 *>(cache->v);
    sp.qs = at<__nv_bfloat16>(ws, w.qs);
    sp.qs_lo = at<__nv_bfloat16>(ws, w.qs_lo);
    sp.ks = at<__nv_bfloat16>(ws, w.ks);
    sp.ks_lo = at<__nv_bfloat16>(ws, w.ks_lo);
    sp.vs = at<__nv_bfloat16>(ws, w.vs);
    sp.err = d_err;
    sp.batch = B;
    sp.n = n;
    sp.R = w.R;
    sp.max_len = max_len;
    sp.rope = rope_turns(layer->rope_theta);
    if (launch_rope_stage(sp, s) != cudaSuccess) return MG_ERR_CUDA;
    qsrc = sp.qs;
    // the precise form streams V in 64-key quarter tiles
    if (!map_rows(&tka, sp.ks, w.R, outer, kTcKeys) || !map_rows(&tkl, sp.ks_lo, w.R, outer, kTcKeys) ||
        !map_rows(&tva, sp.vs, w.R, outer, kTcKeys / 4))
      return MG_ERR_CUDA;
    tkb = tka;
    tvb = tva;
  } else {
    if (!map_cache(&tka, cache, cache->k, kTcKeys) || !map_cache(&tva, cache, cache->v, kTcVRows))
      return MG_ERR_CUDA;
    const uint64_t dims[4] = {static_cast<uint64_t>(kD), kHkv, static_cast<uint64_t>(n),
                              static_cast<uint64_t>(B)};
    const uint32_t kbox[4] = {64, 1, kTcKeys, 1};
    const uint32_t vbox[4] = {64, 1, kTcVRows, 1};
    if (!make_map(&tkb, k_new, 4, dims, kbox) || !make_map(&tvb, v_new, 4, dims, vbox))
      return MG_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(kD), kHq, static_cast<uint64_t>(n),
                              static_cast<uint64_t>(B)};
    const uint32_t box[4] = {64, kGroup, kTcPosPerTile, 1};
    if (!make_map(&tq, qsrc, 4, dims, box)) return MG_ERR_CUDA;
    if (!local) {
      tql = tq;
      tkl = tka;
    } else if (!make_map(&tql, at<__nv_bfloat16>(ws, w.qs_lo), 4, dims, box)) {
      return MG_ERR_CUDA;
    }
  }
  TcParams p;
  p.pos0 = d_pos0;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.part_o = w.splits > 1 ? at<float>(ws, w.part_o) : nullptr;
  p.part_lse = w.splits > 1 ? at<float>(ws, w.part_lse) : nullptr;
  p.err = d_err;
  p.batch = B;
  p.n = n;
  p.kind = layer->kind;
  p.window = local ? kWindow : 0;
  p.staged = local ? 1 : 0;
  p.splits = w.splits;
  p.qblocks = (n + kTcPosPerCta - 1) / kTcPosPerCta;
  p.max_len = max_len;
  p.slots = cache->slots;
  p.scale_log2 = layer->scale * static_cast<float>(M_LOG2E);
  p.map = cache_map(cache);
  if (launch_attn_tc(p, tq, tka, tva, tkb, tvb, tql, tkl, s) != cudaSuccess) return MG_ERR_CUDA;
  if (w.splits > 1) {
    CombineParams c;
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.o = p.o;
    c.rows = B * n * kHq;
    c.splits = w.splits;
    c.overlap = 0;
    return launch_status(launch_combine(c, s));
  }
  return MG_OK;
}

}  // namespace
}  // namespace mg

extern "C" {

int mg_attn_verify(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0, int32_t n,
                   int32_t max_len, const void *q, const void *k_new, const void *v_new, void *o,
                   void *ws, size_t ws_bytes, uint32_t *d_err, void *stream) {
  return block_attention(MG_OP_VERIFY, layer, cache, d_pos0, n, max_len, q, k_new, v_new, o, ws,
                         ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

int mg_attn_prefill(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0,
                    int32_t n, int32_t max_len, const void *q, const void *k_new,
                    const void *v_new, void *o, void *ws, size_t ws_bytes, uint32_t *d_err,
                    void *stream) {
  return block_attention(MG_OP_PREFILL, layer, cache, d_pos0, n, max_len, q, k_new, v_new, o, ws,
                         ws_bytes, d_err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
