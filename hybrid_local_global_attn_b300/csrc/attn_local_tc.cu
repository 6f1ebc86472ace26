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
//  * RoPE by slot, as in the single-token ring kernel: slot s holds position
//    p - ((p - s) mod 2048), so <R(p) q, R(j) k> is <R(b) q, R(s) k> for
//    s <= b and <R(b + 2048) q, R(s) k> for s > b (b = p mod 2048).  A block
//    token k sits at slot (p0 + k) mod 2048 under the same rule.  Keys are
//    rotated in shared memory (ring rows by angles computed before the
//    dependency wait), each query twice into two A operands; the scores of
//    both versions land in TMEM and the softmax picks per (row, key).
//  * Ring slots that the block's tokens up to i are about to overwrite hold
//    positions outside token i's window and are masked, as are slots past
//    the last written position.
//  * Softmax: thread = (row, half of the keys); maxima and sums meet in
//    shared memory; P goes back to TMEM (bf16) as the A operand of P.V.
//  * Cluster merge: CTA r owns head r; every CTA stages its normalised rows
//    and log-sum-exps per owner in shared memory and sends each owner one
//    bulk copy (cp.async.bulk into the owner's shared memory), whose bytes
//    complete on the owner's mbarrier; the owner merges the 16 partials per
//    token.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

constexpr int kPiece = kWindow / kLocCluster;  // 128 ring slots per CTA
constexpr int kBlk = kMaxLocalTokens;          // block rows (first CTA)
constexpr int kKeysMax = kPiece + kBlk;        // 144
constexpr int kTpc = kTcPosPerTile;            // 8 tokens = 128 rows per CTA
constexpr int kThreads = 256;
constexpr int kBoxBytes = kKeysMax * 128;      // one 64-dim box of 144 key rows
constexpr int kKVSmem = 2 * kBoxBytes;         // dims 0-63 box, dims 64-127 box
constexpr int kQBox = kTcRows * 128;           // 16 KB
constexpr int kQSmem = 2 * kQBox;              // one rotated query version
constexpr int kQAngSmem = kTpc * 2 * 64 * 8;   // [token][version][freq] (cos, sin)
constexpr int kRedSmem = 4 * kTcRows * 4;      // [half][m, l][row]
// Inbox of the owning CTA: rows [source][token][128] fp32, then lse
// [source][8 tokens].  One source's rows for one owner are contiguous, so they
// travel as one bulk copy.
constexpr int kInboxRows = kLocCluster * kTpc * kD * 4;  // 64 KB
constexpr int kInboxLse = kLocCluster * kTpc * 4;        // 512 B
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKVSmem;
constexpr int kOffQ = kOffV + kKVSmem;         // version 0, then version 1; staging later
constexpr int kOffQAng = kOffQ + 2 * kQSmem;
constexpr int kOffRed = kOffQAng + kQAngSmem;
constexpr int kOffTurn = kOffRed + kRedSmem;   // 64 turns (uint64)
constexpr int kOffW = kOffTurn + 64 * 8;       // merge weights [token][source]
constexpr int kOffBars = kOffW + kTpc * kLocCluster * 4;
constexpr int kOffInbox = kOffBars + 64;
constexpr int kSmem = kOffInbox + kInboxRows + kInboxLse + 1024;  // + alignment slack
// Staging of this CTA's normalised rows, [owner][token][128] fp32 with the
// owner blocks 16 bytes apart beyond their size (so that the 32 rows a warp
// stores at once fall on different banks), and lse [owner][8]: over the
// query buffers, free once P.V has run.
constexpr int kStageOwner = kTpc * kD * 4 + 16;
constexpr int kOffStage = kOffQ;
constexpr int kOffStageLse = kOffQ + kLocCluster * kStageOwner;
static_assert(kLocCluster * kStageOwner + kInboxLse <= 2 * kQSmem + kQAngSmem,
              "staging fits the query buffers");
// TMEM columns: scores of the two query versions, then O.  P (bf16 pairs)
// overwrites the first 72 columns of the first scores.
constexpr uint32_t kColSlo = 0, kColShi = 160, kColO = 320;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory into
// another CTA's, completing the bytes on that CTA's mbarrier.
__device__ __forceinline__ void bulk_to_cta(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\ncp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred P;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n"
        " selp.u32 %0, 1, 0, P;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (test()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (test()) return true;
    if ((it & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
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
// rotate 8 (x, y) pairs held as bf16 in (lo, hi) by the angles a[0..7]
__device__ __forceinline__ void rot8(uint4 &lo, uint4 &hi, const float2 *a) {
  uint32_t *l = reinterpret_cast<uint32_t *>(&lo);
  uint32_t *h = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x0 = bf16lo(l[e]), x1 = bf16hi(l[e]);
    const float y0 = bf16lo(h[e]), y1 = bf16hi(h[e]);
    const float2 a0 = a[2 * e], a1 = a[2 * e + 1];
    l[e] = pack_bf16x2(x0 * a0.x - y0 * a0.y, x1 * a1.x - y1 * a1.y);
    h[e] = pack_bf16x2(x0 * a0.y + y0 * a0.x, x1 * a1.y + y1 * a1.x);
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    local_tc_kernel(const __grid_constant__ LocalParams p, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + kOffK, sV = sbase + kOffV, sQ = sbase + kOffQ;
  float2 *qang = reinterpret_cast<float2 *>(smem + kOffQAng);
  float *red = reinterpret_cast<float *>(smem + kOffRed);
  float *inbox = reinterpret_cast<float *>(smem + kOffInbox);
  uint64_t *turns = reinterpret_cast<uint64_t *>(smem + kOffTurn);
  float *wts = reinterpret_cast<float *>(smem + kOffW);
  const uint32_t bar_k = sbase + kOffBars, bar_v = bar_k + 8, bar_s = bar_k + 16;
  const uint32_t bar_o = bar_k + 24, bar_inbox = bar_k + 32;

  const int nq = (p.n + kTpc - 1) / kTpc;  // token groups per sequence
  const int g = blockIdx.y, b = blockIdx.z / nq;
  const int i0 = (blockIdx.z % nq) * kTpc;  // first token of this CTA
  const int cnt = min(kTpc, p.n - i0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t my_rank = cluster_rank();
  const int32_t s0 = static_cast<int32_t>(my_rank) * kPiece;
  const int32_t head = b * kHkv + g;
  const bool blk_here = my_rank == 0;  // the first CTA also scores the block rows
  const int nkeys = blk_here ? kKeysMax : kPiece;

  // ---- prologue: kernel parameters only (overlaps the previous kernel) ----
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar_k, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_inbox, 1);
    fence_mbar_init();
    // from each CTA: cnt rows and the lse block
    mbar_arrive_expect_tx(bar_inbox, kLocCluster * (cnt * kD * 4 + kTpc * 4));
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    for (int x = 0; x < 2; ++x) {
      tma_prefetch_l2_3d(&tk, 64 * x, s0, head);
      tma_prefetch_l2_3d(&tv, 64 * x, s0, head);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid < 64) turns[tid] = p.turn[tid];
  __syncthreads();
  // slot angles of this thread's ring row (krow) at frequencies 32 kh .. 32 kh + 31
  const int krow = tid >> 1, kh = tid & 1;
  float2 kang[32];
#pragma unroll
  for (int f = 0; f < 32; ++f) rope_cos_sin(s0 + krow, turns[32 * kh + f], kang[f].x, kang[f].y);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  cluster_arrive_relaxed();
  pdl_wait();
  pdl_launch_dependents();

  // The position is loaded first, but nothing waits for it until the loads
  // that do not depend on it are in flight: the piece's tiles, the raw
  // queries and the block's rows (for an invalid position they are read and
  // then dropped).
  const int32_t p0 = p.pos[b];
  if (tid == 0) {  // the piece's 128 K and V rows
    mbar_arrive_expect_tx(bar_k, kPiece * kRowBytes);
    mbar_arrive_expect_tx(bar_v, kPiece * kRowBytes);
    for (int x = 0; x < 2; ++x) {
      tma_load_3d(sK + x * kBoxBytes, &tk, bar_k, 64 * x, s0, head);
      tma_load_3d(sV + x * kBoxBytes, &tv, bar_v, 64 * x, s0, head);
    }
  }

  // raw query of row qr (token qr / 16, head qr % 16), dims 32 kh.. and 64 + 32 kh..
  const int qr = tid >> 1, qt = qr >> 4;
  uint4 qx[4], qy[4];
  {
    const bool live = qt < cnt;
    const __nv_bfloat16 *src =
        p.q + ((static_cast<size_t>(b) * p.n + i0 + (live ? qt : 0)) * kHq + g * kGroup + (qr & 15)) * kD +
        32 * kh;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      qx[c] = live ? __ldg(reinterpret_cast<const uint4 *>(src) + c) : make_uint4(0u, 0u, 0u, 0u);
      qy[c] = live ? __ldg(reinterpret_cast<const uint4 *>(src + 64) + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // block rows 128..143 of K and V (first CTA): thread tid < 128 takes row
  // tid / 8, 8-dim chunk tid % 8 (and its partner 64 dims on); K rotated by
  // its slot's angle
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
  // query-version angles: entry (t, v, f) = R((b_t + 2048 v) w_f), b_t the slot of token t
  for (int e = tid; e < kTpc * 2 * 64; e += kThreads) {
    const int t = e >> 7, v = (e >> 6) & 1, f = e & 63;
    float2 a = make_float2(1.f, 0.f);
    if (t < cnt && !bad)
      rope_cos_sin(((p0 + i0 + t) & (kWindow - 1)) + kWindow * v, turns[f], a.x, a.y);
    qang[e] = a;
  }
  // which query versions some valid (token, key) pair uses (CTA-uniform)
  bool need_lo = false, need_hi = false;
  if (!bad) {
    for (int t = 0; t < cnt; ++t) {
      const int32_t bt = (p0 + i0 + t) & (kWindow - 1);
      need_lo = need_lo || s0 <= bt;
      need_hi = need_hi || s0 + kPiece - 1 > bt;
    }
    if (blk_here) need_lo = need_hi = true;  // block slots may fall on either side
  }

  if (blk_here && tid < 128) {
    const int k = bk, c = bc;
    if (bad) kx = ky = vx = vy = make_uint4(0u, 0u, 0u, 0u);
    if (k < p.n && !bad) {
      float2 a[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        rope_cos_sin((p0 + k) & (kWindow - 1), turns[8 * c + e], a[e].x, a[e].y);
      rot8(kx, ky, a);
    }
    const uint32_t o = swz(kPiece + k, c);
    sts128(sK + o, kx);
    sts128(sK + kBoxBytes + o, ky);
    sts128(sV + o, vx);
    sts128(sV + kBoxBytes + o, vy);
  }
  __syncthreads();  // query angles ready

  // rotated queries, version v at sQ + v * kQSmem (K-major, 128-byte swizzle)
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    if (v == 0 ? !need_lo : !need_hi) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = 4 * kh + c;  // 8-dim chunk
      uint4 lo = qx[c], hi = qy[c];
      rot8(lo, hi, qang + (qt < kTpc ? qt : 0) * 128 + v * 64 + 8 * cc);
      const uint32_t o = sQ + v * kQSmem + swz(qr, cc);
      sts128(o, lo);
      sts128(o + kQBox, hi);
    }
  }
  // ring keys: once the tile has landed, rotate each row by its slot's angle
  bool ok = mbar_wait(bar_k, 0, &abort_flag);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int cc = 4 * kh + c;
    const uint32_t o = sK + swz(krow, cc);
    uint4 lo = lds128(o), hi = lds128(o + kBoxBytes);
    rot8(lo, hi, kang + 8 * c);
    sts128(o, lo);
    sts128(o + kBoxBytes, hi);
  }
  fence_proxy_async_smem();  // the tensor core reads what the threads wrote
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------ S = Q K^T ----
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idq = idesc_bf16_f32(128, nkeys, 0, 0);
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      if (v == 0 ? !need_lo : !need_hi) continue;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t oq = (kk >> 2) * kQBox + (kk & 3) * 32;
        const uint32_t ok_ = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        mma_ss(tbase + (v == 0 ? kColSlo : kColShi), smem_desc_sw128(sQ + v * kQSmem + oq, 16, 1024),
               smem_desc_sw128(sK + ok_, 16, 1024), idq, kk > 0 ? 1u : 0u);
      }
    }
    mma_commit(bar_s);
  }

  // -------------------------------------------------------------- softmax ----
  // thread: row r (TMEM lane), half hh of the keys (0: keys 0..63; 1: keys
  // 64..127 and the block keys 128..143)
  const int r = 32 * (warp & 3) + lane, hh = warp >> 2;
  const uint32_t lane_bits = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const int rt = r >> 4;                       // token of the row
  const bool row_live = rt < cnt && !bad;
  const int32_t ri = i0 + rt;                  // token index in the block
  const int32_t rp = p0 + ri;                  // its position
  const int32_t rb = rp & (kWindow - 1);       // its slot
  const int32_t rn = min(rp + 1, kWindow);     // slots holding positions
  ok = __all_sync(0xffffffffu, mbar_wait(bar_s, 0, &abort_flag) && ok);
  tc_fence_after();
  const float sl2 = p.scale_log2;
  float sv[80];  // this thread's scores (scaled, masked)
  float mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 2; ++c) {  // ring keys 64 hh + 32 c ..
    const int j0 = 64 * hh + 32 * c;
    uint32_t lo[32], hi[32];
    tmem_ld32(tbase + lane_bits + kColSlo + j0, lo);
    tmem_ld32(tbase + lane_bits + kColShi + j0, hi);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int32_t s = s0 + j0 + j;
      const bool stale = ((s - p0) & (kWindow - 1)) <= ri;  // a block token takes this slot
      const bool valid = row_live && s < rn && !stale;
      const float x = __uint_as_float(s <= rb ? lo[j] : hi[j]) * sl2;
      sv[32 * c + j] = valid ? x : -INFINITY;
      mx = fmaxf(mx, sv[32 * c + j]);
    }
  }
  if (hh == 1) {
#pragma unroll
    for (int j = 0; j < 16; ++j) sv[64 + j] = -INFINITY;
    if (blk_here) {  // block keys k = 0..15 at slots (p0 + k) mod 2048
      uint32_t lo[16], hi[16];
      tmem_ld16(tbase + lane_bits + kColSlo + kPiece, lo);
      tmem_ld16(tbase + lane_bits + kColShi + kPiece, hi);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int32_t sk = (p0 + k) & (kWindow - 1);
        const float x = __uint_as_float(sk <= rb ? lo[k] : hi[k]) * sl2;
        sv[64 + k] = (row_live && k <= ri) ? x : -INFINITY;
        mx = fmaxf(mx, sv[64 + k]);
      }
    }
  }
  red[(2 * hh + 0) * kTcRows + r] = mx;
  __syncthreads();  // every S value is read before P overwrites it
  const float M = fmaxf(red[0 * kTcRows + r], red[2 * kTcRows + r]);
  const float Ms = M == -INFINITY ? 0.f : M;
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
    tmem_st16(tbase + lane_bits + kColSlo + 32 * hh + 16 * c, pk);
  }
  if (hh == 1 && blk_here) {  // block keys: columns 64..71
    uint32_t pk[8];
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
      const float e0 = fast_exp2(sv[64 + k] - Ms), e1 = fast_exp2(sv[64 + k + 1] - Ms);
      l += e0 + e1;
      pk[k >> 1] = pack_bf16x2(e0, e1);
    }
    tmem_st8(tbase + lane_bits + kColSlo + kPiece / 2, pk);
  }
  red[(2 * hh + 1) * kTcRows + r] = l;
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  const float L = red[1 * kTcRows + r] + red[3 * kTcRows + r];

  // ------------------------------------------------------------- O = P V ----
  if (tid == 0) {
    ok = mbar_wait(bar_v, 0, &abort_flag) && ok;
    tc_fence_after();
    const uint32_t idv = idesc_bf16_f32(128, 128, 0, 1);
    for (int kk = 0; kk < nkeys / 16; ++kk)
      mma_ts(tbase + kColO, tbase + kColSlo + 8 * kk,
             smem_desc_sw128(sV + kk * 2048, kBoxBytes, 1024), idv, kk > 0 ? 1u : 0u);
    mma_commit(bar_o);
  }
  ok = __all_sync(0xffffffffu, mbar_wait(bar_o, 0, &abort_flag) && ok && !abort_flag);
  if (!ok && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
  tc_fence_after();

  // ---------------- send this CTA's normalised rows to the owning CTAs ----
  // Stage [owner = head][token][128] and lse [owner][8] over the query
  // buffers (every MMA has retired), then one bulk copy per owner.
  const bool have = ok && row_live && L > 0.f;
  const float inv = have ? 1.f / L : 0.f;
  const int owner = r & 15;
  float *stage = reinterpret_cast<float *>(smem + kOffStage);
  float *stage_lse = reinterpret_cast<float *>(smem + kOffStageLse);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int d0 = 64 * hh + 32 * c;
    uint32_t ov[32];
    tmem_ld32(tbase + lane_bits + kColO + d0, ov);
    tmem_wait_ld();
    float4 *dst = reinterpret_cast<float4 *>(stage + (owner * kStageOwner) / 4 + rt * kD + d0);
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      dst[j / 4] = make_float4(have ? __uint_as_float(ov[j]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 1]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 2]) * inv : 0.f,
                               have ? __uint_as_float(ov[j + 3]) * inv : 0.f);
  }
  if (hh == 0) stage_lse[owner * kTpc + rt] = have ? M + __log2f(L) : -INFINITY;
  fence_proxy_async_smem();  // the bulk copies read what the threads wrote
  tc_fence_before();
  __syncthreads();  // staging complete; TMEM reads done
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  cluster_wait();  // every CTA of the cluster runs, its inbox barrier is set
  if (tid < kLocCluster) {  // thread h sends owner h its rows and lse
    const uint32_t own = static_cast<uint32_t>(tid);
    const uint32_t inbox_s = smem_u32(inbox);
    const uint32_t obar = map_to_rank(bar_inbox, own);
    bulk_to_cta(map_to_rank(inbox_s + my_rank * (kTpc * kD * 4), own),
                sbase + kOffStage + own * kStageOwner, cnt * kD * 4, obar);
    bulk_to_cta(map_to_rank(inbox_s + kInboxRows + my_rank * (kTpc * 4), own),
                sbase + kOffStageLse + own * (kTpc * 4), kTpc * 4, obar);
    bulk_commit_wait_read();  // the staging is not reused, but copies finish reading first
  }

  // ------------- merge the rows this CTA owns (head my_rank of the group) ----
  // (CTA-uniform: the block below has a barrier)
  const bool all_in = __syncthreads_and(mbar_wait_cluster(bar_inbox, 0));
  if (!all_in && tid == 0) set_err(p.err, MG_DERR_TIMEOUT);
  if (all_in) {
    const float *lse = inbox + kInboxRows / 4;  // [source][8]
    if (tid < cnt * kLocCluster) {  // weight of source j for token t, normalised
      const int t = tid >> 4, j = tid & 15;
      float Mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kLocCluster; ++k) Mx = fmaxf(Mx, lse[k * kTpc + t]);
      float den = 0.f;
#pragma unroll
      for (int k = 0; k < kLocCluster; ++k)
        den += (Mx == -INFINITY || lse[k * kTpc + t] == -INFINITY) ? 0.f : fast_exp2(lse[k * kTpc + t] - Mx);
      const float mine = lse[j * kTpc + t];
      wts[t * kLocCluster + j] =
          (den > 0.f && mine != -INFINITY) ? fast_exp2(mine - Mx) / den : 0.f;
    }
    __syncthreads();
    const int d = tid & (kD - 1);
    for (int t = tid >> 7; t < cnt; t += kThreads / kD) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kLocCluster; ++j)
        acc = fmaf(wts[t * kLocCluster + j], inbox[(j * kTpc + t) * kD + d], acc);
      const size_t orow = (static_cast<size_t>(b) * p.n + i0 + t) * kHq + g * kGroup + my_rank;
      p.o[orow * kD + d] = __float2bfloat16_rn(acc);
    }
  }
}

cudaError_t launch_local_tc(const LocalParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                            cudaStream_t s) {
  static_assert(kGroup == kLocCluster, "CTA r of a cluster owns head r of the group");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  if (p.n < 1 || p.n > kMaxLocalTokens || p.batch < 1 || p.k_new == nullptr)
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(local_tc_kernel), kSmem, 3);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kLocCluster, kHkv, p.batch * ((p.n + kTpc - 1) / kTpc));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kLocCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, local_tc_kernel, p, tk, tv);
}

}  // namespace mg
