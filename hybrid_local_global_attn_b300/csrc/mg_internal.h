// mg_internal.h -- constants and kernel parameter blocks shared by the host
// entry points and the kernels of libmg (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "mg.h"

namespace mg {

// Shape fixed by the model: 32 query heads, 2 KV heads, head dim 128, a
// 2048-token window for local layers.
constexpr int kHq = 32;
constexpr int kHkv = 2;
constexpr int kD = 128;
constexpr int kGroup = kHq / kHkv;  // 16 query heads per KV head
constexpr int kWindow = 2048;
constexpr int kRowBytes = kD * 2;   // one bf16 head row
// Hidden size of a token and the projected features (32 q + 2 k + 2 v heads)
constexpr int kHidden = 6656;
constexpr int kQkvFeatures = (kHq + 2 * kHkv) * kD;  // 4608

// Every pipeline wait gives up after this much wall time (ns).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Decode (split-KV flash-decode on mma.sync):
constexpr int kDecTile = 64;              // keys per pipeline stage
constexpr int kDecStages = 3;             // TMA ring depth (2 CTAs per SM)
constexpr int kDecWarps = 4;              // consumer warps, 16 keys each per stage
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one TMA producer warp
constexpr int kDecStageBytes = 2 * kDecTile * kRowBytes;  // K + V
constexpr int kDecMaxSplits = 296;
constexpr int kDecPrefetchTiles = 8;  // L2-prefetched tiles per global-layer CTA
// FP8 (e4m3) global decode: 128-key stages of 32 KB (K codes + transposed V
// codes), 3 deep
constexpr int kE4m3Tile = 128;
constexpr int kE4m3Stages = 3;
constexpr int kE4m3PrefetchTiles = 8;

// Local layers (ring attention for up to 16 query tokens): one 16-CTA cluster
// per (sequence, KV head, group of query tokens), 128 ring slots per CTA.
constexpr int kLocCluster = 16;
constexpr int kMaxLocalTokens = 16;

// tcgen05 attention (verify + prefill): one query tile of 128 rows
// (8 positions x 16 heads) per CTA, key tiles of 256 (S = Q K^T as
// M128 N256 K16 MMAs: the cost of a tcgen05.mma barely depends on N).
constexpr int kTcRows = 128;
constexpr int kTcKeys = 256;
constexpr int kTcVRows = kTcKeys / 2;             // V streams in half tiles
constexpr int kTcPosPerTile = kTcRows / kGroup;   // 8
constexpr int kTcPosPerCta = kTcPosPerTile;       // 8
// Local verify of 2..16 tokens: CTAs per cluster by the number of (sequence,
// KV head, group of 8 tokens) triples -- the fewest rounds per CTA that put
// every cluster in one wave (on this B300 at most 7 clusters of 16 CTAs run
// at once, 15 of 8, 33 of 4).
inline int local_tc_cluster(int64_t triples) { return triples <= 7 ? 16 : triples <= 15 ? 8 : 4; }
constexpr int kTcKStages = 2;                     // K tiles (64 KB)
constexpr int kTcVStages = 2;                     // V half tiles (32 KB)
constexpr int kTcKTileBytes = kTcKeys * kRowBytes;   // 64 KB (two 64-dim boxes)
constexpr int kTcVTileBytes = kTcVRows * kRowBytes;  // 32 KB
constexpr int kTcQBytes = kTcRows * kRowBytes;       // 32 KB
constexpr int kTcSmem =
    kTcQBytes + kTcKStages * kTcKTileBytes + kTcVStages * kTcVTileBytes + 1024 + 256;
constexpr int kTcThreads = 320;  // warps 0-3 / 4-7 softmax of even / odd key tiles, 8 TMA, 9 MMA
constexpr int kTcMaxSplits = 160;

struct RopeTurns {
  uint64_t turn[64];  // w_i / (2 pi) in 0.64 fixed point, w_i = theta^(-2i/128)
};
// Slot steps between the keys one thread of the local kernel rotates.
constexpr int kRopeSteps[3] = {8, 64, 72};

// Where a global layer keeps token position pos of (sequence b, KV head g).
// Linear: row pos of [batch][2][slots][128] (outer index b * 2 + g); paged:
// row pos % page_size of page table[b][pos / page_size] in the pool
// [num_pages][2][page_size][128] (outer index page * 2 + g).  In both
// cases the element offset of the row is (outer * rows + row) * 128, and a
// 3D tensor map (128, rows, outer) reads it at (x, row, outer).
struct CacheMap {
  const int32_t *table;  // nullptr: linear
  int32_t rows;          // slots (linear) or page_size (paged)
  int32_t pages_per_seq, num_pages;
};

#ifdef __CUDACC__
// (row, outer) of position pos; an out-of-range page entry flags
// MG_DERR_PAGE (when err != nullptr) and becomes page 0.
__device__ __forceinline__ void cache_coord(const CacheMap &m, int b, int g, int32_t pos,
                                            int32_t *row, int32_t *outer, uint32_t *err) {
  if (m.table == nullptr) {
    *row = pos;
    *outer = b * 2 + g;
    return;
  }
  int32_t page = m.table[static_cast<size_t>(b) * m.pages_per_seq + pos / m.rows];
  if (page < 0 || page >= m.num_pages) {
    if (err != nullptr) atomicOr(err, MG_DERR_PAGE);
    page = 0;
  }
  *row = pos % m.rows;
  *outer = page * 2 + g;
}
#endif

struct AppendParams {
  const __nv_bfloat16 *k_new, *v_new;  // [B][n][2][128]
  __nv_bfloat16 *k_cache, *v_cache;    // [B][2][slots][128]
  const int32_t *pos0;
  // speculative commit: keep the first count[b] of the n tokens (nullptr:
  // all n) and optionally write pos0[b] + count[b] to pos_next
  const int32_t *count;
  int32_t *pos_next;
  uint32_t *err;
  int32_t batch, n, slots, kind;
  CacheMap map;  // global layers: where each position's row lives
  // MG_E4M3 caches (global, linear): codes of k * k_mul[g], v * v_mul[g]
  // (the reciprocals of power-of-two scales, so exact); V transposed per
  // 64-position tile
  int32_t dtype;
  float k_mul[2], v_mul[2];
};

// A commit into up to MG_COMMIT_MAX_LAYERS caches in one launch; the block
// rows of layer l start l * layer_stride elements after common.k_new/v_new.
struct CommitLayersParams {
  AppendParams common;  // positions, counts, rows of layer 0, batch, n, error word
  __nv_bfloat16 *k_cache[MG_COMMIT_MAX_LAYERS], *v_cache[MG_COMMIT_MAX_LAYERS];
  int32_t slots[MG_COMMIT_MAX_LAYERS], kind[MG_COMMIT_MAX_LAYERS];
  CacheMap map[MG_COMMIT_MAX_LAYERS];
  int32_t dtype[MG_COMMIT_MAX_LAYERS];
  float k_mul[MG_COMMIT_MAX_LAYERS][2], v_mul[MG_COMMIT_MAX_LAYERS][2];
  size_t layer_stride;
  int32_t layers;
};

struct DecodeParams {  // global layers
  const int32_t *pos;
  const __nv_bfloat16 *q;  // [B][32][128]
  // Optional fused append of the query token's own K/V ([B][1][2][128]):
  // when k_new != nullptr the CTA whose split holds the token's slot writes
  // it into the cache before reading that tile.
  const __nv_bfloat16 *k_new, *v_new;
  __nv_bfloat16 *k_cache, *v_cache;
  float *part_o;           // [B][32][splits][128]
  float *part_lse;         // [B][32][splits]   (log2 domain)
  // splits == 1: each CTA writes its rows of o directly (no partials, no
  // combine kernel)
  __nv_bfloat16 *o;        // [B][32][128]
  uint32_t *err;
  int32_t batch, slots, splits, max_len;
  float scale_log2;        // softmax scale * log2(e)
  CacheMap map;            // linear or paged rows of the cache
  float k_scale[2], v_scale[2];  // MG_E4M3 caches: per KV head (powers of two)
  // Failure-detection self-test (bf16 kernel only): limit of the pipeline
  // waits (kWaitLimitNs normally), and the key tile at which the producer
  // stops issuing copies (-1: never), so that the consumers' wait for it runs
  // out.
  uint64_t wait_ns;
  int32_t stall_tile;
  int32_t early;  // 1: position and the first tiles read before the dependency wait
  int32_t overlap;  // 1: with a single split, let the next kernel start at once
};


struct LocalParams {  // local layers, n <= kMaxLocalTokens query tokens
  const int32_t *pos;  // [B]: position of query token 0
  const __nv_bfloat16 *q;  // [B][n][32][128]
  // The block's own K/V ([B][n][2][128]); query i sees tokens 0..i of it in
  // place of the ring rows of their slots.  nullptr: the ring already holds
  // every position the queries see (decode after mg_kv_append).
  const __nv_bfloat16 *k_new, *v_new;
  __nv_bfloat16 *k_cache, *v_cache;  // ring [B][2][2048][128]
  __nv_bfloat16 *o;                  // [B][n][32][128]
  uint32_t *err;
  int32_t batch, n, max_len;
  int32_t write_new;   // 1: also store the block rows into the ring (fused append, n == 1)
  int32_t early;       // 1: position and ring read before the dependency wait (decode, n == 1)
  int32_t overlap;     // 1: let the next kernel start at once (decode, n == 1)
  // local verify (n >= 2): the clusters' exchange buffers in the workspace,
  // rows [cluster][16 heads][cluster size][8 tokens][128] and lse [.][.][.][8]
  float *x_rows, *x_lse;
  float scale_log2;
  uint64_t turn[64];   // as in RopeTurns
  float2 step[3][64];  // (cos, sin) of kRopeSteps[k] * w_i, from double
};

struct CombineParams {
  const float *part_o;    // [rows][splits][128]
  const float *part_lse;  // [rows][splits]
  __nv_bfloat16 *o;       // [rows][128]
  int32_t rows, splits;
  int32_t overlap;        // 1: let the next kernel start at once
};

struct StageParams {
  const int32_t *pos0;
  const __nv_bfloat16 *q;                 // [B][n][32][128]
  const __nv_bfloat16 *k_new, *v_new;     // [B][n][2][128]
  const __nv_bfloat16 *k_cache, *v_cache; // ring [B][2][2048][128]
  __nv_bfloat16 *qs, *qs_lo;              // [B][n][32][128]  rotated q (hi, lo)
  __nv_bfloat16 *ks, *ks_lo, *vs;         // [B][2][R][128]  rows = pos - c0 + 2048
  uint32_t *err;
  int32_t batch, n, R, max_len;
  RopeTurns rope;
};

struct TcParams {
  const int32_t *pos0;
  __nv_bfloat16 *o;  // direct output [B][n][32][128] (splits == 1)
  float *part_o;     // [B*n*32][splits][128] (splits > 1)
  float *part_lse;   // [B*n*32][splits]
  uint32_t *err;
  int32_t batch, n, kind, window, staged, splits, qblocks, max_len, slots;
  float scale_log2;
  // Global layers: rows of the cache.  A paged cache aligns the cache's key
  // tiles to multiples of 256 (so a tile never straddles two pages) and
  // masks the keys of the top tile at or past the block start.
  CacheMap map;
};

struct QkvParams {  // fused QKV projection + append
  const int32_t *pos0;               // [B]: position of each sequence's first token
  __nv_bfloat16 *q_out;              // [B][n][32][128]
  __nv_bfloat16 *k_out, *v_out;      // [B][n][2][128] or nullptr
  __nv_bfloat16 *k_cache, *v_cache;  // the layer's cache (ring, linear or paged)
  float *part;                       // split-K partials [splits][M][4608]
  uint32_t *err;
  int32_t M, n, batch, kind, slots, splits, ksteps;
  CacheMap map;
};

// Launch with programmatic stream serialization, so the kernel may be
// scheduled while the previous kernel in the stream drains; every kernel of
// the library calls pdl_wait() before reading anything an earlier kernel
// wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the kernel's dynamic shared-memory limit once per device (so that no
// attribute call happens while a stream is being captured into a graph).
cudaError_t ensure_smem_attr(const void *kernel, int bytes, int kernel_id);

// Kernel launchers (defined next to each kernel).
cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t s);
cudaError_t launch_kv_commit_layers(const CommitLayersParams &p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t s);
// FP8 cache: tk over K codes (128-byte rows), tv over transposed V tiles
cudaError_t launch_decode_e4m3(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                               cudaStream_t s);
// single-token ring kernel and the tcgen05 ring kernel
// for draft blocks (8 tokens per CTA)
cudaError_t launch_local_tc(const LocalParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t s);
cudaError_t launch_local_attn(LocalParams p, const CUtensorMap &tk, const CUtensorMap &tv,
                              cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t s);
cudaError_t launch_rope_stage(const StageParams &p, cudaStream_t s);
// K-range splits the projection uses for M tokens (1 when the output tiles
// fill the GPU), and the launch (the GEMM, then the split reduction)
int qkv_splits(int32_t M);
cudaError_t launch_qkv(QkvParams p, const CUtensorMap &tx, const CUtensorMap &tw, cudaStream_t s);
// (tql, tkl: the lo halves of staged queries and keys, read by the precise
// form that local layers run)
cudaError_t launch_attn_tc(const TcParams &p, const CUtensorMap &tq, const CUtensorMap &tka,
                           const CUtensorMap &tva, const CUtensorMap &tkb, const CUtensorMap &tvb,
                           const CUtensorMap &tql, const CUtensorMap &tkl, cudaStream_t s);

}  // namespace mg
