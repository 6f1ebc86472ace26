// attn_local_tc.cu -- verify pass of a local (sliding-window, RoPE) layer on
// the tensor cores: up to 8 draft tokens per CTA, read straight from the
// 2048-slot ring cache.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// sections 01 and 04; "Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析",
// section "第三招"): draft token i of a block starting at p0 (position
// p = p0 + i) attends the keys at positions [max(0, p-2047), p] with RoPE:
// the ring holds every position before p0, the block's own tokens p0..p come
// from the caller (the ring is not written).
//
// Design:
//  * One 16-CTA cluster per (sequence, KV head, group of 8 tokens); CTA r
//    takes ring slots [128 r, 128 r + 128), the first CTA also the 16 block
//    rows.  The 8 tokens x 16 heads form one M = 128 tcgen05 tile (row =
//    16 * token + head), so a single Q.K^T (N = 128 or 144 keys) and a
//    single P.V per CTA cover every token.
//  * RoPE relative to the block start.  <R(p0 + i) q, R(j) k> =
//    <R(i) q, R(j - p0) k>: token i's query is rotated by R(i), and each key
//    by its offset from p0 -- a block token k by R(k), ring slot s (which
//    holds position p0 - ((p0 - s) mod 2048)) by R(s - b) for s < b and
//    R(s - b - 2048) for s > b (b = p0 mod 2048; slot b itself holds
//    p0 - 2048, outside every token's window).  R(s) is computed before the
//    dependency wait, R(-b) and R(-b - 2048) once p0 is known.
//  * Precision: rotated queries and keys are kept as bf16 pairs hi =
//    bf16(x), lo = bf16(x - hi), and S accumulates Qhi.Khi + Qhi.Klo +
//    Qlo.Khi (24 MMAs of K = 16 into one TMEM accumulator): the scores carry
//    the rounding of the rotated operands at about 2^-17 of |q||k| instead of
//    2^-9, which keeps sharply peaked softmax rows (large |q|) within
//    tolerance.  The query halves live in TMEM (the A operand), the key
//    halves in shared memory.
//  * Ring slots that the block's tokens up to i are about to overwrite hold
//    positions outside token i's window and are masked, as are slots past
//    the last written position.
//  * Softmax: thread = (row, half of the keys); maxima and sums meet in
//    shared memory; P goes back to TMEM (bf16) as the A operand of P.V.
//  * Cluster merge through L2: each CTA owns 16 / (cluster size) heads;
//    every CTA stages its normalised rows and log-sum-exps in shared memory
//    (a transpose: a thread holds one row), copies them with coalesced
//    stores into its slots of an exchange buffer in the workspace, and one
//    cluster barrier (release / acquire) publishes them; each owner then
//    reads its heads' partials from L2 and merges them per token in
//    registers.  (All-to-all pushes over distributed shared memory -- bulk
//    copies or remote stores -- moved these 64 KB per CTA at ~25 GB/s per SM
//    here, ~3 us per layer; the L2 route takes ~2.)
//  * Cluster size by batch: at most 7 clusters of 16 CTAs run at once on
//    this B300 (a 16-CTA cluster takes 16 SMs of one GPC), 15 of 8, 33 of 4.
//    With more (sequence, KV head, token group) triples than one wave of 16,
//    the window is cut into 8 or 4 pieces and each CTA walks its piece in
//    rounds of 128 slots: S of a round in TMEM, an online softmax (running
//    max; the P.V accumulator in TMEM rescaled when the max moves), the next
//    round's keys loading while a round's softmax runs and V double-buffered.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

constexpr int kPiece = kWindow / kLocCluster;  // 128 ring slots per round
constexpr int kBlk = kMaxLocalTokens;          // block rows (first CTA, first round)
constexpr int kKeysMax = kPiece + kBlk;        // 144
constexpr int kTpc = kTcPosPerTile;            // 8 tokens = 128 rows per CTA
constexpr int kThreads = 256;
constexpr int kBoxBytes = kKeysMax * 128;      // one 64-dim box of 144 key rows
constexpr int kKVSmem = 2 * kBoxBytes;         // dims 0-63 box, dims 64-127 box
constexpr int kAngSmem = 2 * 64 * 8;           // R(-b), R(-b - 2048) per frequency
constexpr int kRedSmem = 4 * kTcRows * 4;      // [half][m, l][row]
// Staging of this CTA's normalised rows, [head][token][128] fp32 with the
// head blocks 16 bytes apart beyond their size (so that the 32 rows a warp
// stores at once fall on different banks), and lse [head][8]: over the key
// buffers, free once the last Q.K^T has run.
constexpr int kStageOwner = kTpc * kD * 4 + 16;
static_assert(kLocCluster * kStageOwner + kLocCluster * kTpc * 4 <= 2 * kKVSmem,
              "staging fits the key buffers");
// Each CTA allocates all 512 TMEM columns, so a second CTA on the same SM
// would wait in tcgen05.alloc: the dynamic shared memory keeps it to one.
constexpr int kOneCtaPerSm = 120 * 1024;

template <int kRounds> struct TcLocPlan {
  static constexpr int kCl = kLocCluster / kRounds;  // CTAs per cluster
  static constexpr int kOwned = kGroup / kCl;        // heads each CTA merges
  static constexpr int kVBufs = kRounds > 1 ? 2 : 1;
  static constexpr int kOffK = 0;                    // rotated keys, hi parts
  static constexpr int kOffKl = kOffK + kKVSmem;     // rotated keys, lo parts
  static constexpr int kOffV = kOffKl + kKVSmem;     // V, one buffer per round in flight
  static constexpr int kOffAng = kOffV + kVBufs * kKVSmem;
  static constexpr int kOffRed = kOffAng + kAngSmem;
  static constexpr int kOffTurn = kOffRed + kRedSmem;  // 64 turns (uint64), then R(128 w_f)
  static constexpr int kOffBars = kOffTurn + 64 * 8 + 64 * 8;
  static constexpr int kOffQ = kOffBars + 64;          // raw queries [128 rows][256 B], swizzled
  static constexpr int kUsed = kOffQ + kTcRows * kD * 2 + 1024;  // + alignment slack
  static constexpr int kSmem = kUsed > kOneCtaPerSm ? kUsed : kOneCtaPerSm;
  static constexpr int kOffStage = kOffK;
  static constexpr int kOffStageLse = kOffK + kLocCluster * kStageOwner;
};
// TMEM columns: scores (P as bf16 pairs overwrites their first 72 columns),
// O, and the rotated queries' hi and lo halves (bf16 pairs, the A operand).
constexpr uint32_t kColS = 0, kColO = 160, kColQh = 288, kColQl = 352;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster: the global writes made before it
// are visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync_release_acquire() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cg_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg_f(const float *p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y);
}
// Two fp32 values as bf16 pairs hi = bf16(v) and lo = bf16(v - hi).
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo(hi), b - bf16hi(hi));
}
// Rotate 8 (x, y) pairs held as bf16 in (x8, y8) -- dims i..i+7 and their
// partners i+64..i+71 -- by the angles a[0..7] in fp32, and split each
// rotated value into bf16 hi and lo parts.
__device__ __forceinline__ void rot8_split(uint4 x8, uint4 y8, const float2 *a, uint4 &xh,
                                           uint4 &xl, uint4 &yh, uint4 &yl) {
  const uint32_t *x = reinterpret_cast<const uint32_t *>(&x8);
  const uint32_t *y = reinterpret_cast<const uint32_t *>(&y8);
  uint32_t *oxh = reinterpret_cast<uint32_t *>(&xh), *oxl = reinterpret_cast<uint32_t *>(&xl);
  uint32_t *oyh = reinterpret_cast<uint32_t *>(&yh), *oyl = reinterpret_cast<uint32_t *>(&yl);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x0 = bf16lo(x[e]), x1 = bf16hi(x[e]);
    const float y0 = bf16lo(y[e]), y1 = bf16hi(y[e]);
    const float2 a0 = a[2 * e], a1 = a[2 * e + 1];
    split2(x0 * a0.x - y0 * a0.y, x1 * a1.x - y1 * a1.y, oxh[e], oxl[e]);
    split2(x0 * a0.y + y0 * a0.x, x1 * a1.y + y1 * a1.x, oyh[e], oyl[e]);
  }
}

}  // namespace

template <int kRounds>
__global__ void __launch_bounds__(kThreads, 1)
    local_tc_kernel(const __grid_constant__ LocalParams p, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  using Plan = TcLocPlan<kRounds>;
  constexpr int kCl = Plan::kCl, kOwned = Plan::kOwned, kVBufs = Plan::kVBufs;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + Plan::kOffK, sKl = sbase + Plan::kOffKl, sV0 = sbase + Plan::kOffV;
  float2 *ang = reinterpret_cast<float2 *>(smem + Plan::kOffAng);
  float *red = reinterpret_cast<float *>(smem + Plan::kOffRed);
  uint64_t *turns = reinterpret_cast<uint64_t *>(smem + Plan::kOffTurn);
  float2 *step_round = reinterpret_cast<float2 *>(smem + Plan::kOffTurn + 64 * 8);  // R(128 w_f)
  const uint32_t bar_k = sbase + Plan::kOffBars, bar_s = bar_k + 8, bar_o = bar_k + 16;
  const uint32_t bar_v = bar_k + 24;  // one per V buffer

  const int nq = (p.n + kTpc - 1) / kTpc;  // token groups per sequence
  const int g = blockIdx.y, b = blockIdx.z / nq;
  const int i0 = (blockIdx.z % nq) * kTpc;  // first token of this CTA
  const int cnt = min(kTpc, p.n - i0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t my_rank = cluster_rank();
  const int32_t s0 = static_cast<int32_t>(my_rank) * (kPiece * kRounds);  // first slot of the piece
  const int32_t head = b * kHkv + g;
  const bool blk_here = my_rank == 0;  // the first CTA also scores the block rows (round 0)
  // thread roles: row r (TMEM lane, also the query row it rotates), half hh
  // of the keys (softmax) and of the query's dims (rotation)
  const int r = 32 * (warp & 3) + lane, hh = warp >> 2;
  const uint32_t lane_bits = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const int rt = r >> 4;  // token of the row
  auto issue_k = [&](int u) {  // the round's 128 ring rows of K, raw, into the hi buffer
    mbar_arrive_expect_tx(bar_k, kPiece * kRowBytes);
    for (int x = 0; x < 2; ++x) tma_load_3d(sK + x * kBoxBytes, &tk, bar_k, 64 * x, s0 + kPiece * u, head);
  };
  auto issue_v = [&](int u) {
    const uint32_t sv = sV0 + (u % kVBufs) * kKVSmem, bv = bar_v + 8 * (u % kVBufs);
    mbar_arrive_expect_tx(bv, kPiece * kRowBytes);
    for (int x = 0; x < 2; ++x) tma_load_3d(sv + x * kBoxBytes, &tv, bv, 64 * x, s0 + kPiece * u, head);
  };

  // ---- prologue: kernel parameters only (overlaps the previous kernel) ----
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar_k, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    for (int i = 0; i < kVBufs; ++i) mbar_init(bar_v + 8 * i, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    for (int x = 0; x < 2; ++x) {
      tma_prefetch_l2_3d(&tk, 64 * x, s0, head);
      tma_prefetch_l2_3d(&tv, 64 * x, s0, head);
    }
  }
  // The raw queries and the block's K/V rows may come from the kernel
  // before this one: only their L2 lines are fetched before the wait.
  if ((tid >> 5) < cnt)
    prefetch_l2(p.q + ((static_cast<size_t>(b) * p.n + i0 + (tid >> 5)) * kHq + g * kGroup) * kD +
                64 * (tid & 31));
  if (blk_here && tid < 4 * p.n)
    prefetch_l2(((tid >> 1) & 1 ? p.v_new : p.k_new) +
                ((static_cast<size_t>(b) * p.n + (tid >> 2)) * kHkv + g) * kD + 64 * (tid & 1));
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid < 64) {
    turns[tid] = p.turn[tid];
    if (kRounds > 1) {
      float cs, sn;
      rope_cos_sin(kPiece, p.turn[tid], cs, sn);
      step_round[(tid & 31) * 2 + (tid >> 5)] = make_float2(cs, sn);
    }
  }
  __syncthreads();
  // slot angles R(s w_f) of this thread's ring row (krow) of round 0 at
  // frequencies 32 kh .. 32 kh + 31, and the query angles R(i w_f) of its
  // query row's token i at frequencies 32 hh .. 32 hh + 31 (neither needs
  // the position)
  const int krow = tid >> 1, kh = tid & 1;
  float2 kang[32], qang[32];
#pragma unroll
  for (int f = 0; f < 32; ++f) {
    rope_cos_sin(s0 + krow, turns[32 * kh + f], kang[f].x, kang[f].y);
    rope_cos_sin(i0 + rt, turns[32 * hh + f], qang[f].x, qang[f].y);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  // The position is loaded first, but nothing waits for it until the loads
  // that do not depend on it are in flight: the first rounds' tiles, the raw
  // queries and the block's rows (for an invalid position they are read and
  // then dropped).
  const int32_t p0 = p.pos[b];
  if (tid == 0) {
    issue_k(0);
    for (int u = 0; u < kVBufs; ++u) issue_v(u);
  }
  int issued_k = 1, issued_v = kVBufs;  // (thread 0's counts)
  // The raw queries of the 8 tokens x 16 heads (32 KB), coalesced (a token's
  // 16 heads are 4 KB in a row), into shared memory: row R = 16 token + head,
  // 16-byte chunk c at c ^ (R mod 16) so that a warp's per-row reads below
  // hit distinct banks.
  const uint32_t sQ = sbase + Plan::kOffQ;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int i = it * kThreads + tid, t = i >> 8, R = i >> 4, c = i & 15;  // t = token
    const uint4 v4 = t < cnt ? __ldg(reinterpret_cast<const uint4 *>(
                                   p.q + ((static_cast<size_t>(b) * p.n + i0 + t) * kHq + g * kGroup + (R & 15)) * kD) + c)
                             : make_uint4(0u, 0u, 0u, 0u);
    sts128(sQ + R * 256 + ((c ^ (R & 15)) << 4), v4);
  }
  // block rows 128..143 of K and V (first CTA): thread tid < 128 takes row
  // tid / 8, 8-dim chunk tid % 8 (and its partner 64 dims on)
  const int bk = tid >> 3, bc = tid & 7;
  uint4 kx = make_uint4(0u, 0u, 0u, 0u), ky = kx, vx = kx, vy = kx;
  if (blk_here && tid < 128 && bk < p.n) {
    const size_t src = ((static_cast<size_t>(b) * p.n + bk) * kHkv + g) * kD + 8 * bc;
    kx = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src));
    ky = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src + 64));
    vx = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src));
    vy = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src + 64));
  }

  // now the position
  const bool bad = p0 < 0 || static_cast<int64_t>(p0) + p.n > p.max_len;
  if (bad && my_rank == 0 && g == 0 && i0 == 0 && tid == 0) set_err(p.err, MG_DERR_POSITION);
  const int32_t b0 = p0 & (kWindow - 1);  // slot of the block start
  if (tid < 128) {  // R(-b w_f) and R(-(b + 2048) w_f) at [f mod 32][f / 32][variant]
    float cs, sn;
    const int f = tid & 63, variant = tid >> 6;
    rope_cos_sin(-(b0 + kWindow * variant), turns[f], cs, sn);
    ang[((f & 31) * 2 + (f >> 5)) * 2 + variant] = make_float2(cs, sn);
  }
  __syncthreads();  // the raw queries are in shared memory
  // rotated query halves into TMEM: row r, dims 32 hh.. (columns 16 hh..)
  // and 64 + 32 hh.. (columns 32 + 16 hh..)
  {
    uint32_t h0[16], l0[16], h1[16], l1[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 xh, xl, yh, yl;
      const int cx = 4 * hh + c, cy = 8 + 4 * hh + c;  // chunks of dims 32 hh + 8 c and 64 + ..
      rot8_split(lds128(sQ + r * 256 + ((cx ^ (r & 15)) << 4)), lds128(sQ + r * 256 + ((cy ^ (r & 15)) << 4)),
                 qang + 8 * c, xh, xl, yh, yl);
      h0[4 * c] = xh.x; h0[4 * c + 1] = xh.y; h0[4 * c + 2] = xh.z; h0[4 * c + 3] = xh.w;
      l0[4 * c] = xl.x; l0[4 * c + 1] = xl.y; l0[4 * c + 2] = xl.z; l0[4 * c + 3] = xl.w;
      h1[4 * c] = yh.x; h1[4 * c + 1] = yh.y; h1[4 * c + 2] = yh.z; h1[4 * c + 3] = yh.w;
      l1[4 * c] = yl.x; l1[4 * c + 1] = yl.y; l1[4 * c + 2] = yl.z; l1[4 * c + 3] = yl.w;
    }
    tmem_st16(tbase + lane_bits + kColQh + 16 * hh, h0);
    tmem_st16(tbase + lane_bits + kColQh + 32 + 16 * hh, h1);
    tmem_st16(tbase + lane_bits + kColQl + 16 * hh, l0);
    tmem_st16(tbase + lane_bits + kColQl + 32 + 16 * hh, l1);
  }
  if (blk_here && tid < 128) {  // block token k at offset k from p0: R(k)
    const int k = bk, c = bc;
    uint4 xh = make_uint4(0u, 0u, 0u, 0u), xl = xh, yh = xh, yl = xh;
    if (k < p.n && !bad) {
      float2 a[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rope_cos_sin(k, turns[8 * c + e], a[e].x, a[e].y);
      rot8_split(kx, ky, a, xh, xl, yh, yl);
    } else {
      vx = vy = xh;
    }
    const uint32_t o = swz(kPiece + k, c);
    sts128(sK + o, xh);
    sts128(sK + kBoxBytes + o, yh);
    sts128(sKl + o, xl);
    sts128(sKl + kBoxBytes + o, yl);
    sts128(sV0 + o, vx);  // the first round's V buffer
    sts128(sV0 + kBoxBytes + o, vy);
  }
  __syncthreads();  // R(-b) tables ready

  // ------------------------------------------------------------- rounds ----
  const bool row_live = rt < cnt && !bad;
  const int32_t ri = i0 + rt;                  // token index in the block
  const int32_t rp = p0 + ri;                  // its position
  const int32_t rn = min(rp + 1, kWindow);     // slots holding positions
  const float sl2 = p.scale_log2;
  bool ok = true;
  float m_run = -INFINITY, l_half = 0.f;  // running max (same in both halves), this half's sum
  for (int u = 0; u < kRounds; ++u) {
    const int32_t rs0 = s0 + kPiece * u;           // first slot of the round
    const bool blk_round = blk_here && u == 0;
    const int nkeys = blk_round ? kKeysMax : kPiece;
    // ring keys: once the round's tile has landed, rotate this thread's row
    // by R(s) R(-b) or R(s) R(-b - 2048) and split it
    {
      float2 a[32];
      // the row's variant; the two halves (kh) and variants of a warp read
      // neighbouring entries (no bank conflicts)
      const float2 *ab = ang + kh * 2 + ((rs0 + krow > b0) ? 1 : 0);
#pragma unroll
      for (int f = 0; f < 32; ++f) a[f] = cmul(kang[f], ab[4 * f]);
      ok = mbar_wait(bar_k, u & 1, &abort_flag) && ok;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = 4 * kh + c;
        const uint32_t o = swz(krow, cc);
        uint4 xh, xl, yh, yl;
        rot8_split(lds128(sK + o), lds128(sK + kBoxBytes + o), a + 8 * c, xh, xl, yh, yl);
        sts128(sK + o, xh);
        sts128(sK + kBoxBytes + o, yh);
        sts128(sKl + o, xl);
        sts128(sKl + kBoxBytes + o, yl);
      }
      if (kRounds > 1)
#pragma unroll
        for (int f = 0; f < 32; ++f) kang[f] = cmul(kang[f], step_round[2 * f + kh]);
    }
    fence_proxy_async_smem();  // the tensor core reads what the threads wrote
    if (u == 0) tmem_wait_st();  // and the rotated queries are in TMEM
    tc_fence_before();
    __syncthreads();

    // ------------------------------- S = Qh Kh^T + Qh Kl^T + Ql Kh^T ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idq = idesc_bf16_f32(128, nkeys, 0, 0);
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint32_t qa = tbase + (part == 2 ? kColQl : kColQh);
        const uint32_t kb = part == 1 ? sKl : sK;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ok_ = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ts(tbase + kColS, qa + 8 * kk, smem_desc_sw128(kb + ok_, 16, 1024), idq,
                 (part > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit(bar_s);
    }
    ok = __all_sync(0xffffffffu, mbar_wait(bar_s, u & 1, &abort_flag) && ok);
    tc_fence_after();
    if (tid == 0 && u + 1 < kRounds) {  // the key buffer is free: the next round's keys
      issue_k(u + 1);
      ++issued_k;
    }

    // ------------------------------------------------------ softmax ----
    // thread: row r, half hh of the keys (0: keys 0..63; 1: keys 64..127
    // and, in the first CTA's first round, the block keys 128..143)
    float sv[80];  // this thread's scores (scaled, masked)
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 2; ++c) {  // ring keys 64 hh + 32 c ..
      const int j0 = 64 * hh + 32 * c;
      uint32_t sc[32];
      tmem_ld32(tbase + lane_bits + kColS + j0, sc);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int32_t sl = rs0 + j0 + j;
        const bool stale = ((sl - p0) & (kWindow - 1)) <= ri;  // a block token takes this slot
        const bool valid = row_live && sl < rn && !stale;
        sv[32 * c + j] = valid ? __uint_as_float(sc[j]) * sl2 : -INFINITY;
        mx = fmaxf(mx, sv[32 * c + j]);
      }
    }
    if (hh == 1) {
#pragma unroll
      for (int j = 0; j < 16; ++j) sv[64 + j] = -INFINITY;
      if (blk_round) {  // block keys k = 0..15
        uint32_t sc[16];
        tmem_ld16(tbase + lane_bits + kColS + kPiece, sc);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          sv[64 + k] = (row_live && k <= ri) ? __uint_as_float(sc[k]) * sl2 : -INFINITY;
          mx = fmaxf(mx, sv[64 + k]);
        }
      }
    }
    red[(2 * hh + 0) * kTcRows + r] = mx;
    __syncthreads();  // every S value is read before P overwrites it
    const float m_new = fmaxf(m_run, fmaxf(red[0 * kTcRows + r], red[2 * kTcRows + r]));
    const float Ms = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - Ms);
    m_run = m_new;
    float l = 0.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {  // P of ring keys 64 hh + 32 c .. : TMEM columns 32 hh + 16 c ..
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float e0 = fast_exp2(sv[32 * c + j] - Ms), e1 = fast_exp2(sv[32 * c + j + 1] - Ms);
        l += e0 + e1;
        pk[j >> 1] = pack_bf16x2(e0, e1);
      }
      tmem_st16(tbase + lane_bits + kColS + 32 * hh + 16 * c, pk);
    }
    if (hh == 1 && blk_round) {  // block keys: columns 64..71
      uint32_t pk[8];
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const float e0 = fast_exp2(sv[64 + k] - Ms), e1 = fast_exp2(sv[64 + k + 1] - Ms);
        l += e0 + e1;
        pk[k >> 1] = pack_bf16x2(e0, e1);
      }
      tmem_st8(tbase + lane_bits + kColS + kPiece / 2, pk);
    }
    l_half = l_half * alpha + l;
    if (u + 1 == kRounds) red[(2 * hh + 1) * kTcRows + r] = l_half;  // read after the P.V barrier
    if (u > 0) {
      // the previous round's P.V has retired: rescale this half's 64
      // columns of O to the new running max, and the V buffer it read is free
      ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (u - 1) & 1, &abort_flag) && ok);
      tc_fence_after();
      if (tid == 0 && u + 1 < kRounds) {
        issue_v(u + 1);
        ++issued_v;
      }
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o32[32];
          tmem_ld32(tbase + lane_bits + kColO + 64 * hh + 32 * c, o32);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o32[j] = __float_as_uint(__uint_as_float(o32[j]) * alpha);
          tmem_st32(tbase + lane_bits + kColO + 64 * hh + 32 * c, o32);
        }
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();

    // ------------------------------------------------------ O += P V ----
    if (tid == 0) {
      ok = mbar_wait(bar_v + 8 * (u % kVBufs), (u / kVBufs) & 1, &abort_flag) && ok;
      tc_fence_after();
      const uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
      const uint32_t sv_ = sV0 + (u % kVBufs) * kKVSmem;
      for (int kk = 0; kk < nkeys / 16; ++kk)
        mma_ts(tbase + kColO, tbase + kColS + 8 * kk,
               smem_desc_sw128(sv_ + kk * 2048, kBoxBytes, 1024), idv, (u > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar_o);
    }
  }
  ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (kRounds - 1) & 1, &abort_flag) && ok && !abort_flag);
  if (!ok && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
  if (tid == 0) {
    // Never leave TMEM or shared memory to work still in flight (after a
    // timeout some of it was not waited for): the last MMAs, and the last
    // copies issued into each buffer, with the full wait limit.
    bool w = mbar_wait(bar_o, (kRounds - 1) & 1, nullptr);
    w = mbar_wait(bar_k, (issued_k - 1) & 1, nullptr) && w;
    for (int u = issued_v - 1; u >= 0 && u >= issued_v - kVBufs; --u)
      w = mbar_wait(bar_v + 8 * (u % kVBufs), (u / kVBufs) & 1, nullptr) && w;
    if (!w) set_err(p.err, MG_DERR_TIMEOUT);
  }
  tc_fence_after();
  const float L = red[1 * kTcRows + r] + red[3 * kTcRows + r];

  // ------------- publish this CTA's normalised rows through the workspace ----
  // Stage [head][token][128] and lse [head][8] over the key buffers (every
  // MMA has retired; a thread holds one row), then copy them with coalesced
  // stores into this CTA's slots of the cluster's exchange buffer:
  // rows [head][source][token][128], lse [head][source][token].
  const bool have = ok && row_live && L > 0.f;
  const float inv = have ? 1.f / L : 0.f;
  const int hd = r & 15;
  float *stage = reinterpret_cast<float *>(smem + Plan::kOffStage);
  float *stage_lse = reinterpret_cast<float *>(smem + Plan::kOffStageLse);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int d0 = 64 * hh + 32 * c;
    uint32_t ov[32];
    tmem_ld32(tbase + lane_bits + kColO + d0, ov);
    tmem_wait_ld();
    float4 *dst = reinterpret_cast<float4 *>(stage + (hd * kStageOwner) / 4 + rt * kD + d0);
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      dst[j / 4] = make_float4(have ? __uint_as_float(ov[j]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 1]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 2]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 3]) * inv : 0.f);
  }
  if (hh == 0) stage_lse[hd * kTpc + rt] = have ? m_run + __log2f(L) : -INFINITY;
  tc_fence_before();
  __syncthreads();  // staging complete; TMEM reads done
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  const size_t cid = static_cast<size_t>(head) * nq + blockIdx.z % nq;  // this cluster
  float *xr = p.x_rows + cid * (kGroup * kCl * kTpc * kD);
  float *xl = p.x_lse + cid * (kGroup * kCl * kTpc);
#pragma unroll 4
  for (int i = tid; i < kGroup * kTpc * (kD / 4); i += kThreads) {
    const int h = i / (kTpc * (kD / 4)), rem = i % (kTpc * (kD / 4));  // rem: token * 32 + d4
    reinterpret_cast<float4 *>(xr + (static_cast<size_t>(h) * kCl + my_rank) * (kTpc * kD))[rem] =
        *reinterpret_cast<const float4 *>(stage + (h * kStageOwner) / 4 + rem * 4);
  }
  if (tid < kGroup * kTpc) xl[((tid / kTpc) * kCl + my_rank) * kTpc + tid % kTpc] = stage_lse[tid];
  // Every CTA of the cluster reaches this barrier (all waits above are
  // bounded), and its partials are visible to the others after it.
  cluster_sync_release_acquire();

  // -- merge the rows this CTA owns (heads kOwned * rank + j of the group) ----
  // thread: (head owned j, token t, 4 dims); the partials come from L2 (.cg:
  // the exchange buffer is rewritten by every call, L1 may hold old lines)
  for (int i = tid; i < kOwned * kTpc * (kD / 4); i += kThreads) {
    const int j = i / (kTpc * (kD / 4)), t = (i / (kD / 4)) % kTpc, d4 = i % (kD / 4);
    if (t >= cnt) continue;
    const int hq = static_cast<int>(my_rank) * kOwned + j;
    float ls[kCl];
    float4 rv[kCl];
#pragma unroll
    for (int c = 0; c < kCl; ++c) {
      ls[c] = ld_cg_f(xl + (hq * kCl + c) * kTpc + t);
      rv[c] = ld_cg_f4(xr + ((static_cast<size_t>(hq) * kCl + c) * kTpc + t) * kD + 4 * d4);
    }
    float Mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kCl; ++c) Mx = fmaxf(Mx, ls[c]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kCl; ++c) {
      const float w = (Mx == -INFINITY || ls[c] == -INFINITY) ? 0.f : fast_exp2(ls[c] - Mx);
      den += w;
      acc.x = fmaf(w, rv[c].x, acc.x);
      acc.y = fmaf(w, rv[c].y, acc.y);
      acc.z = fmaf(w, rv[c].z, acc.z);
      acc.w = fmaf(w, rv[c].w, acc.w);
    }
    const float iv = den > 0.f ? 1.f / den : 0.f;
    const size_t orow = (static_cast<size_t>(b) * p.n + i0 + t) * kHq + g * kGroup + hq;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * iv, acc.y * iv);
    pk.y = pack_bf16x2(acc.z * iv, acc.w * iv);
    reinterpret_cast<uint2 *>(p.o + orow * kD)[d4] = pk;
  }
}

namespace {

template <int kRounds>
cudaError_t launch_local_tc_rounds(const LocalParams &p, const CUtensorMap &tk,
                                   const CUtensorMap &tv, cudaStream_t s, int kernel_id) {
  using Plan = TcLocPlan<kRounds>;
  static_assert(Plan::kSmem <= 227 * 1024, "shared memory");
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(local_tc_kernel<kRounds>),
                                   Plan::kSmem, kernel_id);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Plan::kCl, kHkv, p.batch * ((p.n + kTpc - 1) / kTpc));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Plan::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = Plan::kCl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, local_tc_kernel<kRounds>, p, tk, tv);
}

}  // namespace

cudaError_t launch_local_tc(const LocalParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t s) {
  static_assert(kGroup == kLocCluster, "a 16-CTA cluster gives each CTA one head to merge");
  if (p.n < 1 || p.n > kMaxLocalTokens || p.batch < 1 || p.k_new == nullptr ||
      p.x_rows == nullptr || p.x_lse == nullptr)
    return cudaErrorInvalidValue;
  // One cluster per (sequence, KV head, group of 8 tokens), its size by the
  // number of clusters (the workspace's exchange buffers are sized the same way).
  const int cl = local_tc_cluster(static_cast<int64_t>(p.batch) * kHkv * ((p.n + kTpc - 1) / kTpc));
  if (cl == 16) return launch_local_tc_rounds<1>(p, tk, tv, s, 3);
  if (cl == 8) return launch_local_tc_rounds<2>(p, tk, tv, s, 9);
  return launch_local_tc_rounds<4>(p, tk, tv, s, 10);
}

}  // namespace mg
