/*
 * mg.h -- C ABI of the hybrid local/global grouped-query attention library
 * (libmg.so, hand-written CUDA for sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？"
 *        section 01 "128K 上下文怎么压进 24GB 显存" and section 04
 *        "一前一后的两个问题".
 *   [P2] "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
 *        sections "窄缓存为长上下文留出空间" and "长上下文仍然带来计算开销".
 *   [P4] "Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析",
 *        sections "第二招：混合注意力机制节省显存开销" and
 *        "第三招：D-Flash投机解码实现3倍提速".
 *
 * Fixed shape [P1 §01]: 32 query heads, 2 KV heads, head dim 128; query
 * head h reads KV head h/16.  Layers repeat three local layers (2048-token
 * sliding window, RoPE) and one global layer (full causal history, no
 * RoPE): layer l is global iff l % 4 == 3, giving 39 local and 13 global
 * layers out of 52 [P1 §01; P2 "窄缓存为长上下文留出空间"].
 *
 * Conventions shared by every call:
 *   - All tensors are bf16, row-major, in DEVICE memory owned by the caller.
 *     The library never allocates or frees memory and keeps no state beyond
 *     a host-side cache of TMA descriptors.
 *   - Positions are int32 in DEVICE memory, one per sequence.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream and never synchronise the host.
 *   - Return value: MG_OK (0) on success; a nonzero mg_status when an
 *     argument is rejected on the host, in which case nothing is launched;
 *     MG_ERR_CUDA if a launch failed.
 *   - `d_err` is a DEVICE uint32 the kernels OR error bits into
 *     (MG_DERR_*) instead of trapping: a position outside what `max_len`
 *     or the cache allows is skipped and flagged.  The caller zeroes it and
 *     reads it back whenever it synchronises.
 *   - Softmax uses scale `layer->scale` (1/sqrt(128)); products accumulate
 *     in fp32; outputs are rounded to bf16 (round to nearest even).
 */
#ifndef MG_H
#define MG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MG_HQ 32      /* query heads [P1 §01] */
#define MG_HKV 2      /* KV heads [P1 §01] */
#define MG_D 128      /* head dim [P1 §01] */
#define MG_WINDOW 2048 /* local window = ring slots [P1 §01] */
#define MG_VERIFY_MAX 16 /* draft block [P1 §04; P4 "第三招"] */
#define MG_COMMIT_MAX_LAYERS 64 /* layers one mg_kv_commit_layers call can take */

typedef enum { MG_LOCAL = 0, MG_GLOBAL = 1 } mg_kind;

/* Element type of a KV cache. */
typedef enum { MG_BF16 = 0, MG_E4M3 = 1 } mg_dtype;

typedef enum {
  MG_OP_DECODE = 0,
  MG_OP_VERIFY = 1,
  MG_OP_PREFILL = 2
} mg_op;

typedef enum {
  MG_OK = 0,
  MG_ERR_INVALID = 1,     /* null pointer, bad kind, negative size, ... */
  MG_ERR_UNSUPPORTED = 2, /* window != 2048 for local, bad scale/theta, n out of range */
  MG_ERR_CAPACITY = 3,    /* max_len beyond what the cache can hold */
  MG_ERR_WORKSPACE = 4,   /* ws_bytes smaller than mg_workspace_bytes() */
  MG_ERR_CUDA = 5         /* a CUDA launch or driver call failed */
} mg_status;

/* Bits OR-ed into *d_err by the kernels. */
#define MG_DERR_POSITION 1u /* a device position was negative or beyond max_len / capacity */
#define MG_DERR_TIMEOUT 2u  /* a pipeline wait ran out its time limit; the CTA gave up */
#define MG_DERR_COUNT 4u    /* a commit count was outside [0, n]; that sequence was left as it was */
#define MG_DERR_PAGE 8u     /* a page-table entry was outside [0, num_pages); page 0 was used */

/* One attention layer.  kind = MG_LOCAL requires window == 2048 and a
 * positive rope_theta (10000 is the value used throughout; the pages do not
 * give theta); kind = MG_GLOBAL requires window == 0 and ignores
 * rope_theta (global layers carry no RoPE [P2 "长上下文仍然带来计算开销"]). */
typedef struct {
  int32_t kind;      /* mg_kind */
  int32_t window;    /* 2048 (local) or 0 (global) */
  float rope_theta;  /* local only */
  float scale;       /* softmax scale, > 0 */
} mg_layer;

/* One layer's KV cache.  K is stored verbatim (un-rotated).
 *
 * Linear (page_table == NULL): k and v each hold bf16 [batch][2][slots][128].
 * A local layer has slots == 2048 and keeps position pos in slot pos % 2048,
 * reusing the oldest entry [P2 "窄缓存为长上下文留出空间"]; a global layer
 * keeps position pos in slot pos, so slots is its capacity.
 *
 * Paged (global layers only): k and v each hold a pool of num_pages pages,
 * bf16 [num_pages][2][page_size][128], shared by all sequences of the batch.
 * Sequence b keeps position pos in row pos % page_size of physical page
 * page_table[b * (slots / page_size) + pos / page_size], so sequences of
 * different lengths take only the pages they use (the pages weigh page size
 * and fragmentation against usage [P2 "窄缓存为长上下文留出空间"]).  slots
 * is the per-sequence capacity and a multiple of page_size; page_size is a
 * multiple of 256; page_table is int32 [batch][slots / page_size] in device
 * memory, owned and filled by the caller (entries of positions a call does
 * not touch are never read).  A kernel that meets an entry outside
 * [0, num_pages) flags MG_DERR_PAGE and uses page 0 instead (the result is
 * then wrong, but no memory outside the pool is touched).
 *
 * FP8 (dtype == MG_E4M3; global layers, linear layout, slots a multiple of
 * 64): the cache holds OCP E4M3 codes (round to nearest even, saturated at
 * +-448) of k / k_scale[g] and v / v_scale[g], one scale per KV head, each a
 * positive power of two so that the division is exact; attention reads the
 * codes back as code value x scale (cache quantisation shrinks the cache
 * [P2 "窄缓存为长上下文留出空间"]; half the bytes of bf16).
 *   k : uint8 [batch][2][slots][128]
 *   v : uint8 [batch][2][slots / 64][128][64], i.e. each 64-position tile
 *       transposed (dims x positions); inside a tile, position p sits in
 *       column 16 * ((p % 64) / 16) + c(p % 16), c(j) = 4 * ((j % 8) / 2) +
 *       2 * (j / 8) + j % 2.
 * Only append, commit and decode take an FP8 cache (verify and prefill
 * return MG_ERR_UNSUPPORTED). */
typedef struct {
  void *k;
  void *v;
  int32_t batch;
  int32_t slots;
  const int32_t *page_table; /* NULL: linear layout */
  int32_t page_size;         /* paged: tokens per page, a multiple of 256 */
  int32_t num_pages;         /* paged: pages in each of the k and v pools */
  int32_t dtype;             /* mg_dtype; MG_BF16 unless stated */
  float k_scale[2];          /* MG_E4M3: per KV head, positive powers of two */
  float v_scale[2];
} mg_cache;

/* Host-only.  Bytes of one layer's K+V cache: 2 (K,V) x batch x 2 heads x
 * slots x 128 x 2 bytes, slots = 2048 for MG_LOCAL (capacity is ignored)
 * and capacity for MG_GLOBAL.  Per token per layer this is 1024 bytes
 * [P1 §01].  Returns 0 for a bad kind or a negative size. */
size_t mg_cache_bytes(int32_t kind, int32_t batch, int32_t capacity);

/* Host-only.  Bytes of one global layer's FP8 (MG_E4M3) K+V cache: 2 x
 * batch x 2 heads x capacity x 128 bytes (512 per token).  Returns 0 for a
 * negative size or a capacity that is not a multiple of 64. */
size_t mg_e4m3_cache_bytes(int32_t batch, int32_t capacity);

/* Host-only.  Bytes of one layer's paged K+V pools: 2 (K,V) x num_pages x
 * 2 heads x page_size x 128 x 2 bytes.  Returns 0 for a negative size or a
 * page_size that is not a positive multiple of 256. */
size_t mg_page_pool_bytes(int32_t num_pages, int32_t page_size);

/* Host-only.  Workspace bytes that mg_attn_decode (op MG_OP_DECODE, n = 1),
 * mg_attn_verify (MG_OP_VERIFY, n = draft tokens) or mg_attn_prefill
 * (MG_OP_PREFILL, n = chunk tokens) need for this layer, batch and
 * max_len.  The workspace holds split-KV partials (global decode, global
 * verify), the partial rows the CTAs of a local verify cluster exchange
 * (blocks of 2..16 tokens) and, for local prefill, RoPE-rotated copies of
 * the queries and of the keys in the window; local decode (and a one-token
 * local verify) merges inside a thread-block cluster and needs none.
 * Nothing in a workspace needs
 * initialising.  A global-layer decode with one split per (sequence, KV
 * head) -- large batches -- writes its output directly and needs none.
 * Returns 0 if no workspace is needed, (size_t)-1 for bad arguments. */
size_t mg_workspace_bytes(int32_t op, const mg_layer *layer, int32_t batch,
                          int32_t n, int32_t max_len);

/* Host-only.  Number of kernels one mg_attn_decode / mg_append_decode call
 * launches for this layer, batch and max_len: 1 (a local layer, or a global
 * layer with a single split) or 2 (a global layer: the split pass, then the
 * combine kernel).  Returns -1 for bad arguments. */
int mg_decode_kernel_count(const mg_layer *layer, int32_t batch, int32_t max_len);

/* Static description of a status code. */
const char *mg_status_str(int status);

/* Layer kind of layer index l in the 52-layer stack: MG_GLOBAL iff
 * l % 4 == 3 (three local layers then one global [P1 §01]).  Returns -1
 * for l outside [0, 52). */
int mg_layer_kind(int32_t l);

/*
 * KV append [P1 §01; P2 "窄缓存为长上下文留出空间"].
 * Writes K/V of positions pos0[b] .. pos0[b]+n-1 of every sequence b into
 * the cache, verbatim.  Local: slot = pos % 2048; when n > 2048 only the last
 * 2048 tokens are written (the earlier ones would be overwritten by the ring
 * anyway), so the result equals appending one token at a time.  Global:
 * slot = pos; a position >= slots is skipped and flags MG_DERR_POSITION.
 *   k_new, v_new : bf16 [batch][n][2][128] (device)
 *   d_pos0       : int32 [batch] (device)
 *   n            : 0 <= n; n == 0 is a no-op
 */
int mg_kv_append(const mg_layer *layer, const mg_cache *cache,
                 const int32_t *d_pos0, int32_t n, const void *k_new,
                 const void *v_new, uint32_t *d_err, void *stream);

/*
 * Speculative commit [P1 §04; P4 "第三招：D-Flash投机解码实现3倍提速"]: the
 * main model checks a block of drafted tokens in one mg_attn_verify pass and
 * keeps the longest accepted prefix.  This call writes the first count[b]
 * tokens of the block that verify scored (positions p0[b] .. p0[b]+count[b]-1:
 * the anchor token and the accepted drafts) into the cache and never writes
 * the rejected ones, so rolling a rejected draft back costs nothing and the
 * ring slots it would have reused keep their old keys.  The cache afterwards
 * equals mg_kv_append of those count[b] tokens; count[b] == 0 leaves
 * sequence b as it was.  Acceptance depends on verify's output (through the
 * caller's sampling), so this is a separate call after verify, not part of it.
 *   k_new, v_new : bf16 [batch][n][2][128] (device), the block given to verify
 *   d_pos0       : int32 [batch] (device), the block's first position
 *   d_count      : int32 [batch] (device), tokens to keep; a count outside
 *                  [0, n] skips sequence b and flags MG_DERR_COUNT
 *   d_pos_next   : int32 [batch] (device) or NULL; receives p0[b] + count[b]
 *                  (p0[b] itself when sequence b was skipped).  Must not alias
 *                  d_pos0 (MG_ERR_INVALID): every CTA of a sequence reads p0.
 *   n            : block size, 0 <= n; n == 0 is a no-op
 * Positions are checked as in mg_kv_append (MG_DERR_POSITION).
 */
int mg_kv_commit(const mg_layer *layer, const mg_cache *cache,
                 const int32_t *d_pos0, int32_t n, const int32_t *d_count,
                 const void *k_new, const void *v_new, int32_t *d_pos_next,
                 uint32_t *d_err, void *stream);

/*
 * mg_kv_commit of one verified block into the caches of n_layers layers in a
 * single launch (the block's K/V rows of every layer are kept until the
 * caller knows how many tokens were accepted; one launch instead of one per
 * layer).  The same result as calling mg_kv_commit(&layers[l], &caches[l],
 * d_pos0, n, d_count, k_new + l * batch * n * 256, v_new + ..., d_pos_next,
 * ...) for l = 0 .. n_layers - 1.
 *   layers, caches : host arrays of n_layers entries (1 <= n_layers <=
 *                    MG_COMMIT_MAX_LAYERS); every cache has the same batch
 *   k_new, v_new   : bf16 [n_layers][batch][n][2][128] (device)
 * Other arguments as in mg_kv_commit.
 */
int mg_kv_commit_layers(int32_t n_layers, const mg_layer *layers,
                        const mg_cache *caches, const int32_t *d_pos0,
                        int32_t n, const int32_t *d_count, const void *k_new,
                        const void *v_new, int32_t *d_pos_next,
                        uint32_t *d_err, void *stream);

/*
 * Decode attention for one query token per sequence [P1 §04: decode is
 * autoregressive, one token at a time].  The query of sequence b sits at
 * position p = pos[b]; its own K/V must already be in the cache
 * (mg_kv_append first).  Key set: [max(0, p-2047), p] for a local layer,
 * with RoPE applied to q at p and to each key at its own position;
 * [0, p] for a global layer, no RoPE.  Split-KV: the key set is cut into
 * splits handled by separate CTAs, merged by a log-sum-exp combine kernel
 * (a single split writes the output directly).
 *   q, o     : bf16 [batch][32][128] (device)
 *   max_len  : 1 + the largest pos[b] the caller may pass (sizes the grid
 *              and the workspace); pos[b] >= max_len is skipped + flagged
 *   ws       : device workspace of at least
 *              mg_workspace_bytes(MG_OP_DECODE, layer, batch, 1, max_len)
 */
int mg_attn_decode(const mg_layer *layer, const mg_cache *cache,
                   const int32_t *d_pos, int32_t max_len, const void *q,
                   void *o, void *ws, size_t ws_bytes, uint32_t *d_err,
                   void *stream);

/*
 * Append + decode in one pass: the same result as mg_kv_append of the query
 * token's own K/V (n = 1 at pos[b]) followed by mg_attn_decode, with the
 * append folded into the decode kernel (the CTA that reads the token's slot
 * writes it first).  Same arguments as mg_attn_decode plus
 *   k_new, v_new : bf16 [batch][1][2][128] (device)
 * Global layers flag a position >= slots (MG_DERR_POSITION) and skip it,
 * as mg_kv_append does.
 */
int mg_append_decode(const mg_layer *layer, const mg_cache *cache,
                     const int32_t *d_pos, int32_t max_len, const void *q,
                     const void *k_new, const void *v_new, void *o, void *ws,
                     size_t ws_bytes, uint32_t *d_err, void *stream);

/* flags of mg_append_decode_ex */
#define MG_EARLY_START 1u  /* kernels still running write neither the cache nor d_pos */
#define MG_OVERLAP_NEXT 2u /* the next kernel on the stream may begin at once */

/*
 * mg_append_decode with flags; flags == 0 is mg_append_decode itself (any
 * other bit: MG_ERR_INVALID).  Both flags apply to a local layer with a
 * batch of one sequence (where this call's clusters fit on the GPU beside
 * the previous call's) and to a bf16 global layer on a linear cache (any
 * batch); MG_OVERLAP_NEXT also to a global layer on an FP8 cache.  Other
 * cases ignore them.
 *
 * MG_EARLY_START: the caller promises that no kernel that may still be
 * running when this call's kernels start writes this layer's cache or
 * d_pos.  Those kernels are the one enqueued on `stream` just before this
 * call and, when that kernel came from a call with MG_OVERLAP_NEXT, also
 * every kernel that may still have been running when that call started
 * (and so on back).  With the flag the decode kernels read the position and
 * start their cache loads before their programmatic-dependent-launch wait:
 * a local layer also rotates its ring keys there, a global layer issues its
 * first pipeline stages.  q, k_new and v_new are read, and everything is
 * written, after the wait, so the kernel before may produce them (a
 * projection that leaves the append to this call) or be another layer's
 * attention.  The results equal mg_append_decode's bit for bit when the
 * promise holds; when it does not, they may be wrong (stale cache rows or
 * position) but no access leaves the cache or the buffers passed.
 *
 * MG_OVERLAP_NEXT: this call's last kernel lets the next kernel on `stream`
 * begin at once rather than after its own dependency wait, so that a chain
 * of MG_EARLY_START calls -- the layers of one decode step -- runs each
 * call's loads under the calls before it.  A next kernel that waits before
 * reading anything (a plain call of this library, or any kernel that is not
 * this library's) sees no difference.  A chain must not contain a call that
 * depends on an append of an earlier call of the same chain: decode steps
 * in a row need a kernel without the flag between them (a position update,
 * the next step's projections).
 */
int mg_append_decode_ex(const mg_layer *layer, const mg_cache *cache,
                        const int32_t *d_pos, int32_t max_len, const void *q,
                        const void *k_new, const void *v_new, void *o, void *ws,
                        size_t ws_bytes, uint32_t *d_err, uint32_t flags,
                        void *stream);

/*
 * Fused QKV projection with the KV append in its epilogue: the step before
 * the attention calls.  [P1 §01] gives the hidden size (6656), 32 query heads
 * and 2 KV heads of dimension 128, so each token's hidden state projects to
 * 4096 query and 2 x 256 key / value features; the weight layout is this
 * library's reading (the pages give none).  For the n tokens of sequence b,
 * at positions pos0[b] .. pos0[b]+n-1:
 *   y = x W^T  (bf16 products, fp32 accumulation, rounded once to bf16)
 * with output feature f = 128 h + d of query head h (f < 4096), then
 * 4096 + 128 g + d of key head g, then 4352 + 128 g + d of value head g.
 * The query rows go to q_out; the key and value rows are stored in the
 * layer's cache exactly as mg_kv_append stores k_new / v_new (ring slot
 * pos mod 2048 -- of n > 2048 tokens only the last 2048 -- or row pos of a
 * linear or paged global cache), and also to k_out / v_out when given.
 *   x            : bf16 [batch][n][6656] (device, 16-byte aligned)
 *   w            : bf16 [4608][6656] (device): row f holds output feature f's weights
 *   q_out        : bf16 [batch][n][32][128] (device)
 *   k_out, v_out : bf16 [batch][n][2][128] (device), or both NULL
 *   ws           : >= mg_qkv_workspace_bytes(batch, n) bytes (device; with
 *                  few tokens the K range is split and fp32 partials meet
 *                  there; 0 bytes when the output tiles fill the GPU)
 * bf16 caches only (MG_ERR_UNSUPPORTED for MG_E4M3).  A negative pos0[b], or
 * a global position >= slots, flags MG_DERR_POSITION and that row is not
 * stored (q_out / k_out / v_out are still written).
 */
#define MG_HIDDEN 6656       /* hidden size [P1 §01] */
#define MG_QKV_FEATURES 4608 /* (32 + 2 + 2) x 128 */
size_t mg_qkv_workspace_bytes(int32_t batch, int32_t n);
int mg_qkv_append(const mg_layer *layer, const mg_cache *cache, const int32_t *d_pos0, int32_t n,
                  const void *x, const void *w, void *q_out, void *k_out, void *v_out, void *ws,
                  size_t ws_bytes, uint32_t *d_err, void *stream);

/*
 * Failure-detection self-test of the bounded waits (no counterpart on the
 * pages; test infrastructure exposed through the ABI).  It runs
 * mg_attn_decode of a global layer with a bf16 linear or paged cache, except
 * that in every split the producer stops issuing key-tile copies at tile
 * `stall_tile` (0 = the first tile of the split) and the pipeline waits give
 * up after `wait_ns` nanoseconds (1 .. 2e9) instead of the normal 2 s.  A
 * split with more than stall_tile tiles then waits for a tile that never
 * arrives: its consumers time out, set MG_DERR_TIMEOUT in *d_err, stop, wait
 * (with the full limit) for the copies already issued, and the kernel
 * returns; the context stays usable and o holds undefined values.  Nothing
 * faults, traps or hangs.  Same arguments as mg_attn_decode plus the two
 * above; MG_ERR_UNSUPPORTED for a local layer or an FP8 cache.
 */
int mg_debug_decode_stall(const mg_layer *layer, const mg_cache *cache,
                          const int32_t *d_pos, int32_t max_len, const void *q,
                          void *o, void *ws, size_t ws_bytes, uint32_t *d_err,
                          void *stream, uint64_t wait_ns, int32_t stall_tile);

/*
 * Decode attention without a workspace argument, for callers that cannot
 * allocate device memory: for example a plugin inside a host framework that
 * owns every device buffer and gives plugins none, or a serving loop that
 * must not call cudaMalloc on its hot path and has no spare buffer to lend.
 * The pages have no counterpart to this; it is a packaging of
 * mg_attn_decode, with the same arguments minus ws / ws_bytes and the same
 * results.
 *
 * The split partials live in a fixed device array of MG_NOALLOC_SCRATCH_BYTES
 * inside libmg.so (held by every GPU that loads the library until the process
 * exits).  A call whose mg_workspace_bytes(MG_OP_DECODE, layer, batch, 1,
 * max_len) exceeds it returns MG_ERR_WORKSPACE and launches nothing (at the
 * default split counts no batch needs more than about 2.5 MB: a batch large
 * enough for one split per KV head needs none).  The array is shared by all
 * calls on a device and keeps the last call's contents; nothing in it has to
 * start at zero.  Calls that overlap on the GPU (e.g. on two streams) race on
 * it.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, that device current); make that first call before
 * any stream capture.  The address is kept with the context it was found in;
 * after a device reset (a new primary context) the next call looks it up
 * again, so that call too belongs before any capture.
 */
#define MG_NOALLOC_SCRATCH_BYTES (4u << 20)
int mg_attn_decode_noalloc(const mg_layer *layer, const mg_cache *cache,
                           const int32_t *d_pos, int32_t max_len, const void *q,
                           void *o, uint32_t *d_err, void *stream);

/*
 * Parallel verify of a speculative draft block [P1 §04; P4 "第三招"]:
 * n (1..16) consecutive query tokens at positions p0[b] .. p0[b]+n-1 in
 * one pass.  Query i sees the cached keys before p0 inside its window plus
 * the block's own keys 0..i (causal inside the block).  The block's K/V come
 * in k_new/v_new; the cache is read-only here and must hold positions
 * < p0[b].  Appending the accepted prefix afterwards is the caller's call
 * (mg_kv_append), which keeps a local ring exact when drafts are rejected.
 *   q, o         : bf16 [batch][n][32][128] (device)
 *   k_new, v_new : bf16 [batch][n][2][128] (device)
 *   max_len      : >= 1 + max(p0[b]) + n - 1 (key positions incl. the block)
 *   ws           : >= mg_workspace_bytes(MG_OP_VERIFY, layer, batch, n, max_len)
 */
int mg_attn_verify(const mg_layer *layer, const mg_cache *cache,
                   const int32_t *d_pos0, int32_t n, int32_t max_len,
                   const void *q, const void *k_new, const void *v_new,
                   void *o, void *ws, size_t ws_bytes, uint32_t *d_err,
                   void *stream);

/*
 * Causal chunked prefill [P2 "长上下文仍然带来计算开销": full attention,
 * quadratic in global layers; P4 "第二招"].  Chunk of n tokens at positions
 * c0[b] .. c0[b]+n-1; key set of each query as in decode, taken from the
 * cache (positions < c0[b]) and from the chunk's own k_new/v_new.  The cache
 * is read-only; append the chunk afterwards with mg_kv_append.
 *   q, o         : bf16 [batch][n][32][128] (device)
 *   k_new, v_new : bf16 [batch][n][2][128] (device)
 *   max_len      : >= max(c0[b]) + n
 *   ws           : >= mg_workspace_bytes(MG_OP_PREFILL, layer, batch, n, max_len)
 */
int mg_attn_prefill(const mg_layer *layer, const mg_cache *cache,
                    const int32_t *d_pos0, int32_t n, int32_t max_len,
                    const void *q, const void *k_new, const void *v_new,
                    void *o, void *ws, size_t ws_bytes, uint32_t *d_err,
                    void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MG_H */
