// attn_local.cu -- attention of a local (sliding-window, RoPE) layer for up to
// 16 query tokens per sequence, read straight from the 2048-slot ring cache.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// section 01; "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
// section "窄缓存为长上下文留出空间"): the query at position p attends the keys at
// positions [max(0, p-2047), p], both rotated by RoPE; 16 query heads share
// one KV head.  Decode is one such query; the verify pass of a draft block
// ("深度拆解Muse Glimmer", section 04) is n of them, where query p0+i also
// sees the block's own tokens p0..p0+i.
//
// Design (latency-bound: a window is 1 MB of K/V per KV head):
//  * The ring is cut into 16 fixed pieces of 128 slots; the 16 CTAs of one
//    (sequence, KV head, group of query tokens) form a thread-block cluster,
//    one piece each.  The pieces do not depend on the query position, so a
//    CTA starts its tile copies (TMA, 128-byte swizzle) right after the
//    dependency wait and warms L2 with them before it.  A CTA takes up to
//    eight query tokens in turn, all against the same tiles.
//  * RoPE by slot.  Slot s of the ring holds position j = p - ((p - s) mod
//    2048), i.e. j = p - b + s for s <= b and j = p - b - 2048 + s for s > b,
//    b = p mod 2048.  Since R(p)^T R(j) = R(j - p), the score
//    <R(p) q, R(j) k> equals <R(b) q, R(s) k> (s <= b) or
//    <R(b + 2048) q, R(s) k> (s > b).  So keys are rotated by their slot's
//    angle -- each thread computes the angles of its keys into registers
//    before the dependency wait, while the previous kernel is still
//    running -- and each query is rotated twice, by R(b) and R(b + 2048).
//  * The draft block's own tokens (verify) are a separate 16-row tile
//    handled by the cluster's first CTA: query p0+i scores block token
//    k <= i as <R(i) q, R(k) k_k> (= <R(p0+i) q, R(p0+k) k_k>), and the
//    ring slots those tokens are about to overwrite are masked.  A single
//    new token (decode with fused append) instead replaces the row of its
//    slot in the owning CTA's shared-memory copy, and is written to the
//    ring as well.
//  * Eight consumer warps: warp w computes the scores of 16 keys of one tile
//    (mma.sync m16n8k16, the 16 heads as M, queries rotated once per token
//    into shared memory by the whole CTA), the CTA takes one softmax over
//    its keys (row maxima and sums exchanged in shared memory, the
//    probabilities written there as bf16), and warp w then forms P.V for its
//    own 16 of the 128 output dimensions -- no per-warp partial outputs to
//    merge.  With several tokens per CTA the keys are rotated in shared
//    memory once, by the first token.
//  * Cluster merge: CTA r owns head r of the group; every CTA pushes its
//    normalised partial row and its log-sum-exp for each query into the
//    owner's shared memory with st.async, whose bytes complete on the
//    owner's mbarrier; the owner merges as soon as its own inbox is full
//    (no cluster-wide barrier at the end) and writes the bf16 outputs.
#include <mutex>

#include "mg_internal.h"
#include "mg_ptx.cuh"
#include "mma_frag.cuh"

namespace mg {

namespace {

constexpr int kLocWarps = 8;                      // consumer warps
constexpr int kLocThreads = kLocWarps * 32;
constexpr int kCons = kLocWarps * 32;             // consumer threads
constexpr int kPiece = kWindow / kLocCluster;     // 128 ring slots per CTA
constexpr int kLocTiles = kPiece / kDecTile;      // 2 tiles of 64 slots
constexpr int kBlk = kMaxLocalTokens;             // rows of the block tile
constexpr int kTileSmem = kLocTiles * kDecStageBytes;  // K + V of the piece
constexpr int kBlkSmem = 2 * kBlk * kRowBytes;         // K + V of the block
constexpr int kBlkTabSmem = kBlk * 64 * 8;        // (cos, sin) of k w_i, k < 16
constexpr int kQRow = kD + 8;                     // padded bf16 row of a rotated query
constexpr int kQRotSmem = 3 * kGroup * kQRow * 2;  // R(b) q, R(b + 2048) q, R(i) q
constexpr int kPRow = kPiece + kBlk + 8;          // padded bf16 row of P
constexpr int kPSmem = kGroup * kPRow * 2;
constexpr int kQAngSmem = 2 * 64 * 8;
constexpr int kRedSmem = 2 * kLocWarps * kGroup * 4;
constexpr int kConstSmem = 64 * 8 + 64 * 8;       // turns, step of 8 slots
constexpr int kInboxPerToken = (kLocCluster * kD + kLocCluster) * 4;  // o rows, then lse
constexpr int kOffBlk = kTileSmem;
constexpr int kOffBlkTab = kOffBlk + kBlkSmem;
constexpr int kOffQRot = kOffBlkTab + kBlkTabSmem;
constexpr int kOffP = kOffQRot + (kQRotSmem + 255) / 256 * 256;
constexpr int kOffQAng = kOffP + (kPSmem + 255) / 256 * 256;
constexpr int kOffRed = kOffQAng + kQAngSmem;
constexpr int kOffConst = kOffRed + kRedSmem;
constexpr int kOffBars = kOffConst + kConstSmem;
constexpr int kOffInbox = kOffBars + 64;
// dynamic shared memory for `tpc` query tokens per CTA (+ alignment slack)
constexpr int loc_smem_bytes(int tpc) { return kOffInbox + tpc * kInboxPerToken + 1024; }

// Rotate the packed bf16 pairs (lo = dims i,i+1; hi = dims i+64,i+65) by the
// angles of frequencies i and i+1, in fp32, rounding back to bf16.
__device__ __forceinline__ void rot_pair(uint32_t &lo, uint32_t &hi, float2 a0, float2 a1) {
  const float x0 = bf16lo(lo), x1 = bf16hi(lo);
  const float y0 = bf16lo(hi), y1 = bf16hi(hi);
  lo = pack_bf16x2(x0 * a0.x - y0 * a0.y, x1 * a1.x - y1 * a1.y);
  hi = pack_bf16x2(x0 * a0.y + y0 * a0.x, x1 * a1.y + y1 * a1.x);
}

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
// Remote store into another CTA's shared memory that completes its bytes on
// that CTA's mbarrier (both addresses from mapa).
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float a, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr),
               "f"(a), "r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n"
      " selp.u32 %0, 1, 0, P;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (kWaitLimitNs) for phase `parity` of an mbarrier completed by
// other CTAs of the cluster.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory");
}

// Frequency index of table entry f (0..15) of the thread at quad position tq:
// the mma fragments give a thread dimensions 16 ks + 8 h8 + 2 tq + e with
// f = 4 ks + 2 h8 + e (and the partners 64 further on).
__device__ __forceinline__ int freq_of(int f, int tq) {
  return (f >> 2) * 16 + 8 * ((f >> 1) & 1) + 2 * tq + (f & 1);
}

__device__ __forceinline__ void zero4(float (&a)[4]) { a[0] = a[1] = a[2] = a[3] = 0.f; }

}  // namespace

__global__ void __launch_bounds__(kLocThreads, 1)
    local_attn_kernel(const __grid_constant__ LocalParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float2 *blktab = reinterpret_cast<float2 *>(smem + kOffBlkTab);  // [16 k][64 freq]
  uint32_t *pmat = reinterpret_cast<uint32_t *>(smem + kOffP);  // [16 rows][kPRow/2] bf16 pairs
  float2 *qang = reinterpret_cast<float2 *>(smem + kOffQAng);  // [2 versions][64]
  float *red_m = reinterpret_cast<float *>(smem + kOffRed);    // [8 warps][16 rows]
  float *red_l = red_m + kLocWarps * kGroup;
  uint64_t *turns = reinterpret_cast<uint64_t *>(smem + kOffConst);
  float2 *step8 = reinterpret_cast<float2 *>(smem + kOffConst + 64 * 8);
  float *inbox = reinterpret_cast<float *>(smem + kOffInbox);  // [tpc][16 sources][128], lse
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t blk_base = smem_base + kOffBlk;    // K box 0/1 (2 KB each), then V
  const uint32_t qrot_base = smem_base + kOffQRot;  // [3 versions][16 rows][kQRow] bf16
  const uint32_t bar_full = smem_u32(smem + kOffBars);  // 2 tiles
  const uint32_t bar_inbox = bar_full + 8 * kLocTiles;   // the pushes into this CTA's inbox

  const int nq = (p.n + p.tpc - 1) / p.tpc;  // token groups per sequence
  const int g = blockIdx.y;
  const int b = blockIdx.z / nq;
  const int i0 = (blockIdx.z % nq) * p.tpc;  // first query token of this CTA
  const int cnt = min(p.tpc, p.n - i0);     // query tokens of this CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int th = warp >> 2, ws = warp & 3;  // consumer warp: tile and 16-key slice
  const uint32_t my_rank = cluster_rank();
  const int32_t s0 = static_cast<int32_t>(my_rank) * kPiece;
  const int32_t head = b * kHkv + g;  // (sequence, KV head) index of the cache
  const bool has_new = p.k_new != nullptr;
  const bool block_mode = has_new && p.n > 1;  // draft block: separate tile
  const bool patch_mode = has_new && p.n == 1;  // one new token: replaces its ring row
  const bool blk_here = block_mode && my_rank == 0;

  // ---- prologue: reads only kernel parameters, so it overlaps the previous
  // kernel under programmatic dependent launch ----
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int t = 0; t < kLocTiles; ++t) mbar_init(bar_full + 8 * t, 1);
    mbar_init(bar_inbox, 1);
    fence_mbar_init();
    // every CTA of the cluster pushes one row and one lse per query token
    mbar_arrive_expect_tx(bar_inbox, cnt * kInboxPerToken);
  }
  if (threadIdx.x < 64) {
    turns[threadIdx.x] = p.turn[threadIdx.x];
    step8[threadIdx.x] = p.step[0][threadIdx.x];
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    for (int t = 0; t < kLocTiles; ++t)
      for (int x = 0; x < 2; ++x) {
        tma_prefetch_l2_3d(&tk, 64 * x, s0 + t * kDecTile, head);
        tma_prefetch_l2_3d(&tv, 64 * x, s0 + t * kDecTile, head);
      }
  }
  __syncthreads();
  // Slot angles of this thread's 2 keys (slots sb and sb + 8) at its 16
  // frequencies, kept in registers until the keys are rotated: entry
  // 16 sel + f.
  float2 tab[32];
  {
    const int tid = threadIdx.x;
    const int32_t sb = s0 + th * kDecTile + ws * 16 + gr;
#pragma unroll
    for (int f = 0; f < 16; ++f) {
      const int fr = freq_of(f, tq);
      rope_cos_sin(sb, turns[fr], tab[f].x, tab[f].y);
      const float2 r = step8[fr];
      tab[16 + f] = make_float2(tab[f].x * r.x - tab[f].y * r.y, tab[f].y * r.x + tab[f].x * r.y);
    }
    if (blk_here) {  // R(k) for the block offsets k = 0..15
      for (int e = tid; e < kBlk * 64; e += kCons) {
        float cs, sn;
        rope_cos_sin(e >> 6, turns[e & 63], cs, sn);
        blktab[e] = make_float2(cs, sn);
      }
    }
  }
  // First half of a cluster barrier whose wait (before the first store into
  // another CTA's shared memory) proves every CTA of the cluster is running.
  cluster_arrive_relaxed();
  pdl_wait();
  pdl_launch_dependents();

  // The position is loaded first, but nothing below waits for it until the
  // loads that do not depend on it are in flight: the piece's tiles, the
  // block's rows and the raw query (for an invalid position they are read
  // and then dropped).
  const int32_t p0 = p.pos[b];  // position of query token 0 of the sequence

  if (threadIdx.x == 0) {  // the piece's two tiles
    for (int t = 0; t < kLocTiles; ++t) {
      const uint32_t dst = smem_base + t * kDecStageBytes;
      const uint32_t fb = bar_full + 8 * t;
      const int32_t row = s0 + t * kDecTile;
      mbar_arrive_expect_tx(fb, kDecStageBytes);
      tma_load_3d(dst, &tk, fb, 0, row, head);
      tma_load_3d(dst + 8192, &tk, fb, 64, row, head);
      tma_load_3d(dst + 16384, &tv, fb, 0, row, head);
      tma_load_3d(dst + 24576, &tv, fb, 64, row, head);
    }
  }
  if (blk_here) {
    // The block's K/V rows (zeros past the last token): thread t carries
    // 16-byte chunk t % 16 of row t / 16, of both K and V.  Visible to all
    // after the first barrier below.
    const int k = threadIdx.x >> 4, c = threadIdx.x & 15;
    uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
    if (k < p.n) {
      const size_t src = ((static_cast<size_t>(b) * p.n + k) * kHkv + g) * kD;
      kr = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src) + c);
      vr = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src) + c);
    }
    const uint32_t addr = blk_base + (c >> 3) * (kBlk * 128) + sw128(k, c & 7);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(kr.x), "r"(kr.y),
                 "r"(kr.z), "r"(kr.w)
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr + 2 * kBlk * 128),
                 "r"(vr.x), "r"(vr.y), "r"(vr.z), "r"(vr.w)
                 : "memory");
  }
  const bool bad = p0 < 0 || static_cast<int64_t>(p0) + p.n > p.max_len;
  {
    // ---------------------------------------------------- consumer warps ----
    const int tid = threadIdx.x;
    const int32_t key0 = s0 + th * kDecTile + ws * 16;  // first slot of this warp's 16 keys
    const uint32_t kbase = smem_base + th * kDecStageBytes;
    const uint32_t k_row = ws * 16 + ((lane >> 4) << 3) + (lane & 7);
    const uint32_t k_chi = (lane >> 3) & 1;
    // A-fragment row addresses (ldmatrix x4 of a 16 x 16 bf16 block)
    const uint32_t a_row = ((lane & 7) + 8 * ((lane >> 3) & 1));
    const uint32_t p_addr = smem_u32(pmat) + a_row * (kPRow * 2) + 16 * (lane >> 4);
    const uint32_t q_addr = qrot_base + a_row * (kQRow * 2) + 16 * (lane >> 4);
    const uint32_t v_sub = (((lane >> 3) & 1) << 3) + (lane & 7);
    const uint32_t v_chunk = 2 * warp + (lane >> 4);  // this warp's 16 output dims
    const uint32_t inbox_s = smem_u32(inbox);
    // cooperative query rotation: row qr, frequencies 8 qc .. 8 qc + 7
    const int qr = (tid & 127) >> 3, qc = tid & 7;
    bool waited = false, ok = true, rotated = false;

    uint4 qx = make_uint4(0u, 0u, 0u, 0u), qy = qx;  // raw dims 8 qc.. and 64 + 8 qc..
    auto load_q = [&](int i) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + (((static_cast<size_t>(b) * p.n + i) * kHq + g * kGroup) + qr) * kD + 8 * qc);
      qx = __ldg(src);
      qy = __ldg(src + 8);
    };
    load_q(i0);  // needs no position: issued before anything waits for it
    if (bad && my_rank == 0 && g == 0 && i0 == 0 && tid == 0) set_err(p.err, MG_DERR_POSITION);

    // fused append of a single new token: the warp whose keys hold its slot
    const int32_t slot_new = p0 & (kWindow - 1);
    const bool patch_here = patch_mode && !bad && slot_new >= key0 && slot_new < key0 + 16;
    uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
    if (patch_mode) {  // the row's address needs no position; only patch_here uses it
      const size_t src = (static_cast<size_t>(b) * kHkv + g) * kD;
      new_row = lane < 16 ? __ldg(reinterpret_cast<const uint4 *>(p.k_new + src) + (lane & 15))
                          : __ldg(reinterpret_cast<const uint4 *>(p.v_new + src) + (lane & 15));
    }

    for (int t = 0; t < cnt; ++t) {
      const int i = i0 + t;
      const int32_t pq = p0 + i;                        // query position
      const int32_t n_slots = bad ? 0 : min(pq + 1, kWindow);
      const int32_t bq = pq & (kWindow - 1);            // its slot
      float oacc[2][4];
      zero4(oacc[0]);
      zero4(oacc[1]);
      float lse0 = -INFINITY, lse1 = -INFINITY;
      if (s0 < n_slots) {  // CTA-uniform: the piece holds keys of this query
        const bool need_lo = s0 <= bq, need_hi = s0 + kPiece - 1 > bq;
        // (cos, sin) of bq w_f and (bq + 2048) w_f: one per thread
        if (tid < 128) {
          float cs, sn;
          rope_cos_sin(bq + kWindow * (tid >> 6), turns[tid & 63], cs, sn);
          qang[tid] = make_float2(cs, sn);
        }
        consumers_sync();
        // rotated queries: version 0 = R(bq) q, 1 = R(bq + 2048) q, 2 = R(i) q
        {
          const float x[8] = {bf16lo(qx.x), bf16hi(qx.x), bf16lo(qx.y), bf16hi(qx.y),
                              bf16lo(qx.z), bf16hi(qx.z), bf16lo(qx.w), bf16hi(qx.w)};
          const float y[8] = {bf16lo(qy.x), bf16hi(qy.x), bf16lo(qy.y), bf16hi(qy.y),
                              bf16lo(qy.z), bf16hi(qy.z), bf16lo(qy.w), bf16hi(qy.w)};
          auto emit = [&](int v, const float2 *ang) {
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 a0 = ang[2 * e], a1 = ang[2 * e + 1];
              lo[e] = pack_bf16x2(x[2 * e] * a0.x - y[2 * e] * a0.y,
                                  x[2 * e + 1] * a1.x - y[2 * e + 1] * a1.y);
              hi[e] = pack_bf16x2(x[2 * e] * a0.y + y[2 * e] * a0.x,
                                  x[2 * e + 1] * a1.y + y[2 * e + 1] * a1.x);
            }
            const uint32_t dst = qrot_base + (v * kGroup + qr) * (kQRow * 2) + 16 * qc;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(lo[0]),
                         "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 128), "r"(hi[0]),
                         "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                         : "memory");
          };
          if (tid < 128) {
            if (need_lo) emit(0, qang + 8 * qc);
            if (blk_here) emit(2, blktab + i * 64 + 8 * qc);
          } else if (need_hi) {
            emit(1, qang + 64 + 8 * qc);
          }
        }
        if (t + 1 < cnt) load_q(i + 1);  // the next query's loads overlap this one
        consumers_sync();

        if (!waited) {  // tiles (and block rows) in shared memory
          bool w = mbar_wait(bar_full, 0, &abort_flag);
          w = mbar_wait(bar_full + 8, 0, &abort_flag) && w;
          ok = __all_sync(0xffffffffu, w) && !abort_flag;
          if (!ok && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
          waited = true;
          if (patch_here && ok) {
            // the new token's row replaces the ring row of its slot: lane c
            // writes 16-byte chunk c of K (c < 16) or of V
            const uint32_t r = static_cast<uint32_t>(slot_new - s0 - th * kDecTile);
            const int c = lane & 15;
            const uint32_t addr = kbase + (lane < 16 ? 0 : 16384) + (c >> 3) * 8192 + sw128(r, c & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(new_row.x),
                         "r"(new_row.y), "r"(new_row.z), "r"(new_row.w)
                         : "memory");
            if (p.write_new) {
              const size_t dst = (static_cast<size_t>(head) * kWindow + slot_new) * kD;
              reinterpret_cast<uint4 *>((lane < 16 ? p.k_cache : p.v_cache) + dst)[c] = new_row;
            }
            __syncwarp();
          }
        }
        // On a timeout the warp still runs every step below (shared-memory
        // reads only, so it stays in bounds) to keep the named barriers
        // matched, and drops its result.

        // -------------------------------------------------- S = Q K^T ----
        // ring keys: slot s is valid if it holds a position of the window and
        // is not one a block token is about to overwrite
        float sacc[2][2][4];  // [ring, block][n8 tile][fragment]
        {
          const bool use_lo = key0 <= bq, use_hi = key0 + 15 > bq;
          float acc[2][2][2][4];  // [lo / hi query][dims 0-63 / 64-127][n8 tile]
#pragma unroll
          for (int v = 0; v < 2; ++v)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              zero4(acc[v][h][0]);
              zero4(acc[v][h][1]);
            }
          // all fragment loads first, then the rotation and the MMAs
          uint32_t lo[4][4], hi[4][4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t off = sw128(k_row, 2 * ks + k_chi);
            ldsm_x4(kbase + off, lo[ks][0], lo[ks][1], lo[ks][2], lo[ks][3]);
            ldsm_x4(kbase + 8192 + off, hi[ks][0], hi[ks][1], hi[ks][2], hi[ks][3]);
          }
          uint32_t qa[2][4][4], qb[2][4][4];  // [version][ks]: dims 16 ks.. and 64 + 16 ks..
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            if (v == 0 ? use_lo : use_hi) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint32_t a = q_addr + v * (kGroup * kQRow * 2) + 32 * ks;
                ldsm_x4(a, qa[v][ks][0], qa[v][ks][1], qa[v][ks][2], qa[v][ks][3]);
                ldsm_x4(a + 128, qb[v][ks][0], qb[v][ks][1], qb[v][ks][2], qb[v][ks][3]);
              }
            }
          }
          if (!rotated) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
              for (int h8 = 0; h8 < 2; ++h8)
#pragma unroll
                for (int sel = 0; sel < 2; ++sel) {
                  const int j = 16 * sel + 4 * ks + 2 * h8;
                  rot_pair(lo[ks][2 * sel + h8], hi[ks][2 * sel + h8], tab[j], tab[j + 1]);
                }
              if (cnt > 1) {  // later queries read the rotated keys (this warp's own rows)
                const uint32_t off = sw128(k_row, 2 * ks + k_chi);
                stsm_x4(kbase + off, lo[ks][0], lo[ks][1], lo[ks][2], lo[ks][3]);
                stsm_x4(kbase + 8192 + off, hi[ks][0], hi[ks][1], hi[ks][2], hi[ks][3]);
              }
            }
          }
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            if (v == 0 ? !use_lo : !use_hi) continue;  // never read: its scores are not selected
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              mma_16816(acc[v][0][0], qa[v][ks], lo[ks][0], lo[ks][1]);
              mma_16816(acc[v][0][1], qa[v][ks], lo[ks][2], lo[ks][3]);
              mma_16816(acc[v][1][0], qb[v][ks], hi[ks][0], hi[ks][1]);
              mma_16816(acc[v][1][1], qb[v][ks], hi[ks][2], hi[ks][3]);
            }
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int32_t key = key0 + 8 * j + 2 * tq + (e & 1);
              const bool stale = block_mode && ((key - p0) & (kWindow - 1)) <= i;
              const float sv = key <= bq ? acc[0][0][j][e] + acc[0][1][j][e]
                                         : acc[1][0][j][e] + acc[1][1][j][e];
              sacc[0][j][e] = (key < n_slots && !stale) ? sv * p.scale_log2 : -INFINITY;
            }
        }
        // block keys k = 0..15 (first CTA, warp 0): valid for k <= i
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[1][j][e] = -INFINITY;
        const bool blk_warp = blk_here && warp == 0;
        if (blk_warp) {
          float acc[2][2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            zero4(acc[h][0]);
            zero4(acc[h][1]);
          }
          const uint32_t kr = ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t lo[4], hi[4];
            const uint32_t off = sw128(kr, 2 * ks + k_chi);
            ldsm_x4(blk_base + off, lo[0], lo[1], lo[2], lo[3]);
            ldsm_x4(blk_base + kBlk * 128 + off, hi[0], hi[1], hi[2], hi[3]);
            if (!rotated) {
#pragma unroll
              for (int h8 = 0; h8 < 2; ++h8)
#pragma unroll
                for (int sel = 0; sel < 2; ++sel) {
                  const int f = freq_of(4 * ks + 2 * h8, tq);
                  const int kk = gr + 8 * sel;  // block key of this fragment
                  rot_pair(lo[2 * sel + h8], hi[2 * sel + h8], blktab[kk * 64 + f],
                           blktab[kk * 64 + f + 1]);
                }
              if (cnt > 1) {
                stsm_x4(blk_base + off, lo[0], lo[1], lo[2], lo[3]);
                stsm_x4(blk_base + kBlk * 128 + off, hi[0], hi[1], hi[2], hi[3]);
              }
            }
            uint32_t qa[4], qb[4];
            ldsm_x4(q_addr + 2 * (kGroup * kQRow * 2) + 32 * ks, qa[0], qa[1], qa[2], qa[3]);
            ldsm_x4(q_addr + 2 * (kGroup * kQRow * 2) + 128 + 32 * ks, qb[0], qb[1], qb[2], qb[3]);
            mma_16816(acc[0][0], qa, lo[0], lo[1]);
            mma_16816(acc[0][1], qa, lo[2], lo[3]);
            mma_16816(acc[1][0], qb, hi[0], hi[1]);
            mma_16816(acc[1][1], qb, hi[2], hi[3]);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kk = 8 * j + 2 * tq + (e & 1);
              sacc[1][j][e] = kk <= i ? (acc[0][j][e] + acc[1][j][e]) * p.scale_log2 : -INFINITY;
            }
        }
        rotated = true;  // the tiles now hold rotated keys (when cnt > 1)

        // ------------------------------------------------------ softmax ----
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            mx0 = fmaxf(mx0, fmaxf(sacc[u][j][0], sacc[u][j][1]));
            mx1 = fmaxf(mx1, fmaxf(sacc[u][j][2], sacc[u][j][3]));
          }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (tq == 0) {
          red_m[warp * kGroup + gr] = mx0;
          red_m[warp * kGroup + gr + 8] = mx1;
        }
        consumers_sync();
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kLocWarps; ++w) {
          M0 = fmaxf(M0, red_m[w * kGroup + gr]);
          M1 = fmaxf(M1, red_m[w * kGroup + gr + 8]);
        }
        const float Ms0 = M0 == -INFINITY ? 0.f : M0, Ms1 = M1 == -INFINITY ? 0.f : M1;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (u == 1 && !blk_warp) break;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float e0 = fast_exp2(sacc[u][j][0] - Ms0), e1 = fast_exp2(sacc[u][j][1] - Ms0);
            const float e2 = fast_exp2(sacc[u][j][2] - Ms1), e3 = fast_exp2(sacc[u][j][3] - Ms1);
            l0 += e0 + e1;
            l1 += e2 + e3;
            // key column in P: ring keys by slot, then the block keys
            const int kc = (u == 0 ? th * kDecTile + ws * 16 : kPiece) + 8 * j + 2 * tq;
            pmat[gr * (kPRow / 2) + kc / 2] = pack_bf16x2(e0, e1);
            pmat[(gr + 8) * (kPRow / 2) + kc / 2] = pack_bf16x2(e2, e3);
          }
        }
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (tq == 0) {
          red_l[warp * kGroup + gr] = l0;
          red_l[warp * kGroup + gr + 8] = l1;
        }
        consumers_sync();
        float L0 = 0.f, L1 = 0.f;
#pragma unroll
        for (int w = 0; w < kLocWarps; ++w) {
          L0 += red_l[w * kGroup + gr];
          L1 += red_l[w * kGroup + gr + 8];
        }
        // ------------------------------- O[:, 16 w .. 16 w + 16) = P V ----
        float pacc[2][2][4];  // [k-step parity][n8 tile]
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          zero4(pacc[u][0]);
          zero4(pacc[u][1]);
        }
        constexpr int kKk = kPiece / 16;  // ring k-steps; one more for the block
        uint32_t pa[kKk + 1][4], vb[kKk + 1][4];
#pragma unroll
        for (int kk = 0; kk < kKk; ++kk) {
          ldsm_x4(p_addr + kk * 32, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]);
          ldsm_x4_t(smem_base + (kk >> 2) * kDecStageBytes + 16384 + (v_chunk >> 3) * 8192 +
                        sw128(16 * (kk & 3) + v_sub, v_chunk & 7),
                    vb[kk][0], vb[kk][1], vb[kk][2], vb[kk][3]);
        }
        if (blk_here) {
          ldsm_x4(p_addr + kKk * 32, pa[kKk][0], pa[kKk][1], pa[kKk][2], pa[kKk][3]);
          ldsm_x4_t(blk_base + 2 * kBlk * 128 + (v_chunk >> 3) * (kBlk * 128) +
                        sw128(v_sub, v_chunk & 7),
                    vb[kKk][0], vb[kKk][1], vb[kKk][2], vb[kKk][3]);
        }
#pragma unroll
        for (int kk = 0; kk < kKk; ++kk) {
          mma_16816(pacc[kk & 1][0], pa[kk], vb[kk][0], vb[kk][1]);
          mma_16816(pacc[kk & 1][1], pa[kk], vb[kk][2], vb[kk][3]);
        }
        if (blk_here) {
          mma_16816(pacc[kKk & 1][0], pa[kKk], vb[kKk][0], vb[kKk][1]);
          mma_16816(pacc[kKk & 1][1], pa[kKk], vb[kKk][2], vb[kKk][3]);
        }
        if (ok && L0 > 0.f && L1 > 0.f) {
          const float i0f = 1.f / L0, i1f = 1.f / L1;
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            oacc[n][0] = (pacc[0][n][0] + pacc[1][n][0]) * i0f;
            oacc[n][1] = (pacc[0][n][1] + pacc[1][n][1]) * i0f;
            oacc[n][2] = (pacc[0][n][2] + pacc[1][n][2]) * i1f;
            oacc[n][3] = (pacc[0][n][3] + pacc[1][n][3]) * i1f;
          }
          lse0 = M0 + __log2f(L0);
          lse1 = M1 + __log2f(L1);
        }
      }
      // ------------ push this query's partial rows to the CTAs that own them ----
      if (t == 0) cluster_wait();  // every CTA of the cluster runs, its inbox barrier is set
      const uint32_t box_s = inbox_s + t * kInboxPerToken;
      const uint32_t bar0 = map_to_rank(bar_inbox, gr), bar1 = map_to_rank(bar_inbox, gr + 8);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int d = 16 * warp + 8 * n + 2 * tq;
        const uint32_t a = box_s + 4 * (my_rank * kD + d);
        st_async_f32x2(map_to_rank(a, gr), oacc[n][0], oacc[n][1], bar0);
        st_async_f32x2(map_to_rank(a, gr + 8), oacc[n][2], oacc[n][3], bar1);
      }
      if (warp == 0 && tq == 0) {
        const uint32_t a = box_s + 4 * (kLocCluster * kD + my_rank);
        st_async_f32(map_to_rank(a, gr), lse0, bar0);
        st_async_f32(map_to_rank(a, gr + 8), lse1, bar1);
      }
    }
    // never leave the CTA with copies in flight
    if (!waited && threadIdx.x == 0) {
      bool w = mbar_wait(bar_full, 0, nullptr);
      w = mbar_wait(bar_full + 8, 0, nullptr) && w;
      if (!w) set_err(p.err, MG_DERR_TIMEOUT);
    }
  }

  // ------------- merge the rows this CTA owns (head my_rank of the group) ----
  // Every push into this CTA has landed once its inbox barrier completes;
  // the CTA reads and writes no other CTA's memory after its own pushes.
  const bool all_in = mbar_wait_cluster(bar_inbox, 0);
  if (!all_in && threadIdx.x == 0) set_err(p.err, MG_DERR_TIMEOUT);
  if (all_in) {
    const int d = threadIdx.x & (kD - 1);
    for (int t = threadIdx.x >> 7; t < cnt; t += kCons / kD) {
      const float *box = inbox + t * (kInboxPerToken / 4);
      const float *lse = box + kLocCluster * kD;
      float M = -INFINITY;
#pragma unroll
      for (int j = 0; j < kLocCluster; ++j) M = fmaxf(M, lse[j]);
      float acc = 0.f, den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int j = 0; j < kLocCluster; ++j) {
          const float w = lse[j] == -INFINITY ? 0.f : fast_exp2(lse[j] - M);
          den += w;
          acc = fmaf(w, box[j * kD + d], acc);
        }
      }
      const size_t orow = (static_cast<size_t>(b) * p.n + i0 + t) * kHq + g * kGroup + my_rank;
      p.o[orow * kD + d] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
    }
  }
}

namespace {

cudaLaunchConfig_t local_config(int batch, int n, int tpc, cudaStream_t s, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kLocCluster, kHkv, batch * ((n + tpc - 1) / tpc));
  cfg.blockDim = dim3(kLocThreads);
  cfg.dynamicSmemBytes = loc_smem_bytes(tpc);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kLocCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Clusters of the local kernel the device runs at once with `tpc` tokens per
// CTA (queried once per device and tpc; 8 if the query fails).
int max_active_clusters(int tpc) {
  static std::mutex mu;
  static int cache[64][kLocMaxTpc + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  std::lock_guard<std::mutex> lk(mu);
  int &c = cache[dev][tpc];
  if (c == 0) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = local_config(1, 1, tpc, nullptr, attr);
    cfg.numAttrs = 2;
    int num = 0;
    c = (cudaOccupancyMaxActiveClusters(&num, local_attn_kernel, &cfg) == cudaSuccess && num > 0)
            ? num : 8;
  }
  return c;
}

}  // namespace

cudaError_t launch_local_attn(LocalParams p, const CUtensorMap &tk, const CUtensorMap &tv,
                              cudaStream_t s) {
  static_assert(kGroup == kLocCluster, "CTA r of a cluster owns head r of the group");
  static_assert(loc_smem_bytes(kLocMaxTpc) <= 227 * 1024, "shared memory");
  if (p.n < 1 || p.n > kMaxLocalTokens || p.batch < 1) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(local_attn_kernel),
                                   loc_smem_bytes(kLocMaxTpc), 2);
  if (e != cudaSuccess) return e;
  // Tokens per CTA: the fewest that let every cluster run in one wave (each
  // CTA takes its tokens in turn, so more tokens per CTA cost time too).
  p.tpc = kLocMaxTpc;
  for (int tpc = 1; tpc <= kLocMaxTpc; ++tpc) {
    const int clusters = p.batch * kHkv * ((p.n + tpc - 1) / tpc);
    if (clusters <= max_active_clusters(tpc)) {
      p.tpc = tpc;
      break;
    }
    if (tpc >= p.n) {
      p.tpc = tpc;
      break;
    }
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = local_config(p.batch, p.n, p.tpc, s, attr);
  return cudaLaunchKernelEx(&cfg, local_attn_kernel, p, tk, tv);
}

}  // namespace mg
