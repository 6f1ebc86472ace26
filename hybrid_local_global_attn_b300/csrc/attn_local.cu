// attn_local.cu -- attention of one query token per sequence in a local
// (sliding-window, RoPE) layer, read straight from the 2048-slot ring cache:
// decode, and the verify pass of a one-token block.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// section 01; "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
// section "窄缓存为长上下文留出空间"): the query at position p attends the keys at
// positions [max(0, p-2047), p], both rotated by RoPE; 16 query heads share
// one KV head.
//
// Design (latency-bound: a window is 1 MB of K/V per KV head):
//  * The ring is cut into 16 fixed pieces of 128 slots; the 16 CTAs of one
//    (sequence, KV head) form a thread-block cluster, one piece each.  The
//    pieces do not depend on the query position, so a CTA starts its tile
//    copies (TMA, 128-byte swizzle) right after the dependency wait and
//    warms L2 with them before it.
//  * RoPE relative to the query.  <R(p) q, R(j) k> = <q, R(j - p) k>, so the
//    query enters the products exactly as stored and each key is rotated by
//    its offset d = j - p.  Slot s holds j = p - ((p - s) mod 2048), so
//    d = s - b for s <= b and d = s - b - 2048 for s > b (b = p mod 2048).
//    R(d) is composed from the slot angle R(s) -- each thread computes those
//    of its keys before the dependency wait, while the previous kernel is
//    still running -- and R(-b) or R(-b - 2048), 64 frequencies each, which
//    the CTA computes once the position is known; the key in the query's own
//    slot (d = 0) enters unrotated.
//  * Early start (MG_EARLY_START, batch 1): when the caller
//    promises that no kernel still running writes the ring or the
//    positions, the position, the tiles, R(-b) and the rotated key
//    fragments are all ready before the dependency wait; the query and the
//    new row are read after it, the new key entering the fragments as is.
//    With MG_OVERLAP_NEXT the kernel lets the next one begin at once, so
//    that in a chain of such calls each layer's part before the wait runs
//    under the layers before it.
//  * Precision: the rotated key k' is kept as two bf16 values, hi = bf16(k')
//    and lo = bf16(k' - hi), and Q.K^T accumulates q.hi + q.lo (two
//    mma.sync m16n8k16 per fragment, fp32 accumulate).  The score then
//    carries the rounding of k' at about 2^-17 of |q||k| instead of 2^-9: a
//    single bf16 rounding of the rotated key moves a score by ~0.04 when the
//    scaled scores spread by ~40, enough to shift a sharply peaked softmax
//    row by several 1e-2.
//  * Eight consumer warps: warp w computes the scores of 16 keys of one
//    64-slot tile, the CTA takes one softmax over its 128 keys (row maxima
//    and sums exchanged in shared memory, the probabilities written there as
//    bf16), and warp w then forms P.V for its own 16 of the 128 output
//    dimensions.
//  * A single new token (decode with fused append, or the block of a
//    one-token verify) replaces the ring row of its slot in the owning CTA's
//    shared-memory copy; decode also writes it to the ring.
//  * Cluster merge: each CTA owns 16 / (cluster size) heads of the group;
//    every CTA pushes its normalised partial rows and log-sum-exps into the
//    owners' shared memory with st.async, whose bytes complete on the
//    owner's mbarrier; an owner merges as soon as its own inbox is full (no
//    cluster-wide barrier at the end) and writes the bf16 output.
//  * Cluster size by batch: a 16-CTA cluster needs 16 SMs of one GPC, so at
//    most 7 run at once.  With more (sequence, KV head) pairs than that, the
//    window is cut into 8 or 4 pieces of 256 or 512 slots and each CTA walks
//    its piece in rounds of 128 slots (2 tiles): the next round's copies are
//    in flight while a round computes, and an online softmax (running max,
//    rescaled sum and output) carries the rounds.  15 clusters of 8 or 33 of
//    4 run at once.
#include "mg_internal.h"
#include "mg_ptx.cuh"
#include "mma_frag.cuh"

namespace mg {

namespace {

constexpr int kLocWarps = 8;                      // consumer warps
constexpr int kLocThreads = kLocWarps * 32;
constexpr int kRound = 128;                       // ring slots per round (2 tiles)
constexpr int kLocTiles = kRound / kDecTile;      // 2 tiles of 64 slots per round
constexpr int kRoundSmem = kLocTiles * kDecStageBytes;  // K + V of a round
constexpr int kPRow = kRound + 8;                 // padded bf16 row of P
constexpr int kPSmem = kGroup * kPRow * 2;
static_assert(kPSmem >= kGroup * kD * 2, "the P buffer holds the query tile before the first softmax");
constexpr int kAngSmem = 2 * 64 * 8;              // R(-b), R(-b - 2048) per frequency
constexpr int kRedSmem = 2 * kLocWarps * kGroup * 4;
constexpr int kConstSmem = 3 * 64 * 8;            // turns, step of 8 slots, step of a round

// Shared-memory plan of the kernel whose CTAs take `kRounds` rounds (cluster
// of 16 / kRounds CTAs): round buffers, P, the R(-b) table, reductions,
// constants, barriers, then the inbox [heads owned][sources][128] + lse
// [heads owned][sources].
template <int kRounds> struct LocPlan {
  static constexpr int kCl = kLocCluster / kRounds;  // CTAs per cluster
  static constexpr int kHeadsOwned = kGroup / kCl;   // heads each CTA merges
  static constexpr int kSlots = kRound * kRounds;    // ring slots per CTA
  static constexpr int kBufs = kRounds < 2 ? kRounds : 2;
  static constexpr int kInboxBytes = kHeadsOwned * kCl * (kD + 1) * 4;
  static constexpr int kOffP = kBufs * kRoundSmem;
  static constexpr int kOffAng = kOffP + (kPSmem + 255) / 256 * 256;
  static constexpr int kOffRed = kOffAng + kAngSmem;
  static constexpr int kOffConst = kOffRed + kRedSmem;
  static constexpr int kOffBars = kOffConst + kConstSmem;
  static constexpr int kOffInbox = kOffBars + 64;
  static constexpr int kSmem = kOffInbox + kInboxBytes + 1024;  // + alignment slack
};

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y);
}

// Two fp32 values as bf16 pairs hi = bf16(v) and lo = bf16(v - hi).
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo(hi), b - bf16hi(hi));
}

// Rotate the packed bf16 pairs x = (dims i, i+1) and y = (dims i+64, i+65)
// by the angles of frequencies i and i+1 in fp32, and split each rotated
// value into bf16 hi and lo parts.
__device__ __forceinline__ void rot_split(uint32_t x, uint32_t y, float2 a0, float2 a1,
                                          uint32_t &xh, uint32_t &xl, uint32_t &yh,
                                          uint32_t &yl) {
  const float x0 = bf16lo(x), x1 = bf16hi(x);
  const float y0 = bf16lo(y), y1 = bf16hi(y);
  split2(x0 * a0.x - y0 * a0.y, x1 * a1.x - y1 * a1.y, xh, xl);
  split2(x0 * a0.y + y0 * a0.x, x1 * a1.y + y1 * a1.x, yh, yl);
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
  asm volatile("bar.sync 1, %0;" ::"n"(kLocThreads) : "memory");
}

// Frequency index of table entry f (0..15) of the thread at quad position tq:
// the mma fragments give a thread dimensions 16 ks + 8 h8 + 2 tq + e with
// f = 4 ks + 2 h8 + e (and the partners 64 further on).
__device__ __forceinline__ int freq_of(int f, int tq) {
  return (f >> 2) * 16 + 8 * ((f >> 1) & 1) + 2 * tq + (f & 1);
}

__device__ __forceinline__ void zero4(float (&a)[4]) { a[0] = a[1] = a[2] = a[3] = 0.f; }

}  // namespace

template <int kRounds>
__global__ void __launch_bounds__(kLocThreads, 1)
    local_attn_kernel(const __grid_constant__ LocalParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv) {
  using Plan = LocPlan<kRounds>;
  constexpr int kCl = Plan::kCl, kOwned = Plan::kHeadsOwned, kBufs = Plan::kBufs;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint32_t *pmat = reinterpret_cast<uint32_t *>(smem + Plan::kOffP);  // [16 rows][kPRow/2] bf16 pairs
  float2 *ang = reinterpret_cast<float2 *>(smem + Plan::kOffAng);    // [2 versions][64]
  float *red_m = reinterpret_cast<float *>(smem + Plan::kOffRed);    // [8 warps][16 rows]
  float *red_l = red_m + kLocWarps * kGroup;
  uint64_t *turns = reinterpret_cast<uint64_t *>(smem + Plan::kOffConst);
  float2 *step8 = reinterpret_cast<float2 *>(smem + Plan::kOffConst + 64 * 8);
  float2 *step_round = step8 + 64;                                    // R(128 w_f)
  float *inbox = reinterpret_cast<float *>(smem + Plan::kOffInbox);  // [owned][sources][128], lse
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_u32(smem + Plan::kOffBars);  // [buffer][tile]
  const uint32_t bar_inbox = bar_full + 8 * kBufs * kLocTiles; // the pushes into this CTA's inbox

  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int th = warp >> 2, ws = warp & 3;  // tile and 16-key slice of this warp in a round
  const uint32_t my_rank = cluster_rank();
  const int32_t s0 = static_cast<int32_t>(my_rank) * Plan::kSlots;  // this CTA's first slot
  const int32_t head = b * kHkv + g;  // (sequence, KV head) index of the cache
  const bool patch_mode = p.k_new != nullptr;  // the token's own row comes from k_new / v_new
  // the round's two tiles into buffer u % kBufs
  auto issue_round = [&](int u) {
    const uint32_t buf = smem_base + (u % kBufs) * kRoundSmem;
    for (int t = 0; t < kLocTiles; ++t) {
      const uint32_t dst = buf + t * kDecStageBytes;
      const uint32_t fb = bar_full + 8 * ((u % kBufs) * kLocTiles + t);
      const int32_t row = s0 + u * kRound + t * kDecTile;
      mbar_arrive_expect_tx(fb, kDecStageBytes);
      tma_load_3d(dst, &tk, fb, 0, row, head);
      tma_load_3d(dst + 8192, &tk, fb, 64, row, head);
      tma_load_3d(dst + 16384, &tv, fb, 0, row, head);
      tma_load_3d(dst + 24576, &tv, fb, 64, row, head);
    }
  };
  auto wait_round = [&](int u, const volatile int *abort) -> bool {
    bool w = true;
    for (int t = 0; t < kLocTiles; ++t)
      w = mbar_wait(bar_full + 8 * ((u % kBufs) * kLocTiles + t), (u / kBufs) & 1, abort) && w;
    return w;
  };

  // Early start (single-round kernel, caller's promise that no kernel still
  // running writes the ring or the positions): the position, the ring
  // tiles, the R(-b) table and the rotated keys are all prepared before the
  // dependency wait; only the query and the new row -- which an earlier
  // kernel may produce -- are read after it.
  bool early = false, overlap = false;
  if constexpr (kRounds == 1) {
    early = p.early != 0;
    overlap = p.overlap != 0;
  }
  // MG_OVERLAP_NEXT: the next kernel may begin at once, its part before the
  // dependency wait then running under this whole kernel
  if (overlap) pdl_launch_dependents();

  // ---- prologue: reads only kernel parameters (and, with the early start,
  // the ring), so it overlaps the previous kernel under programmatic
  // dependent launch ----
  if (tid == 0) {
    abort_flag = 0;
    for (int t = 0; t < kBufs * kLocTiles; ++t) mbar_init(bar_full + 8 * t, 1);
    mbar_init(bar_inbox, 1);
    fence_mbar_init();
    // every CTA of the cluster pushes one row and one lse per owned head
    mbar_arrive_expect_tx(bar_inbox, Plan::kInboxBytes);
    if (early) issue_round(0);  // the piece does not depend on the position
  }
  if (tid < 64) {
    turns[tid] = p.turn[tid];
    step8[tid] = p.step[0][tid];
    if (kRounds > 1) {
      float cs, sn;
      rope_cos_sin(kRound, p.turn[tid], cs, sn);
      step_round[tid] = make_float2(cs, sn);
    }
  }
  // The query rows and the new token's K/V rows may come from the kernel
  // before this one: only their L2 lines are fetched before the wait.
  if (warp == 1) {
    prefetch_l2(p.q + (static_cast<size_t>(b) * kHq + g * kGroup) * kD + 64 * lane);
    if (patch_mode && lane < 4)
      prefetch_l2((lane < 2 ? p.k_new : p.v_new) + (static_cast<size_t>(b) * kHkv + g) * kD + 64 * (lane & 1));
  }
  if (tid == 0 && !early) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    for (int t = 0; t < kBufs * kLocTiles; ++t)
      for (int x = 0; x < 2; ++x) {
        tma_prefetch_l2_3d(&tk, 64 * x, s0 + t * kDecTile, head);
        tma_prefetch_l2_3d(&tv, 64 * x, s0 + t * kDecTile, head);
      }
  }
  __syncthreads();
  // Slot angles R(s w_f) of this thread's 2 keys of round 0 (slots sb and
  // sb + 8) at its 16 frequencies: entry 16 sel + f; each later round's
  // slots are kRound further on.
  const int32_t key_in_round = th * kDecTile + ws * 16;  // this warp's first slot in a round
  float2 tab[32];
#pragma unroll
  for (int f = 0; f < 16; ++f) {
    const int fr = freq_of(f, tq);
    rope_cos_sin(s0 + key_in_round + gr, turns[fr], tab[f].x, tab[f].y);
    tab[16 + f] = cmul(tab[f], step8[fr]);
  }
  // First half of a cluster barrier whose wait (before the first store into
  // another CTA's shared memory) proves every CTA of the cluster is running.
  cluster_arrive_relaxed();
  if (!early) {
    pdl_wait();
    if (!overlap) pdl_launch_dependents();
  }

  // The position is loaded first, but nothing below waits for it until the
  // loads that do not depend on it are in flight: the first rounds' tiles,
  // the query and the new row (for an invalid position they are read and
  // then dropped).
  const int32_t pq = p.pos[b];
  if (tid == 0 && !early)
    for (int u = 0; u < kBufs; ++u) issue_round(u);
  int issued = kBufs;  // rounds whose copies went out (thread 0's count)
  // Q fragments (A operand, 16 heads x 128 dims)
  uint32_t qf[8][4];
  uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
  const size_t new_src = (static_cast<size_t>(b) * kHkv + g) * kD;  // the new row of (b, g)
  // The group's 16 query rows (4 KB): one coalesced 16-byte load per thread
  // into shared memory (the P buffer, unused until the first softmax; rows
  // 256 bytes apart, 16-byte chunks XOR-swizzled by the row), then ldmatrix
  // into the A fragments -- far sooner ready than 32 scattered 4-byte loads
  // per thread.
  auto load_query = [&]() {
    const int qr = tid >> 4, qc = tid & 15;
    const uint4 v4 = __ldg(reinterpret_cast<const uint4 *>(
                               p.q + (static_cast<size_t>(b) * kHq + g * kGroup + qr) * kD) + qc);
    const uint32_t qs = smem_u32(pmat);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qs + qr * 256 + ((qc ^ (qr & 7)) << 4)),
                 "r"(v4.x), "r"(v4.y), "r"(v4.z), "r"(v4.w)
                 : "memory");
    if (patch_mode)  // the row's address needs no position; only the owning warp uses it
      new_row = lane < 16 ? __ldg(reinterpret_cast<const uint4 *>(p.k_new + new_src) + (lane & 15))
                          : __ldg(reinterpret_cast<const uint4 *>(p.v_new + new_src) + (lane & 15));
    consumers_sync();
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int chunk = 2 * ks + (lane >> 4);
      ldsm_x4(qs + row * 256 + ((chunk ^ (row & 7)) << 4), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  };
  if (!early) load_query();

  const bool bad = pq < 0 || pq >= p.max_len;
  const int32_t n_slots = bad ? 0 : min(pq + 1, kWindow);
  const int32_t bq = pq & (kWindow - 1);  // the query's slot
  const int32_t rounds = s0 >= n_slots ? 0 : min(kRounds, (n_slots - s0 + kRound - 1) / kRound);
  const uint32_t k_row = ws * 16 + ((lane >> 4) << 3) + (lane & 7);
  const uint32_t k_chi = (lane >> 3) & 1;
  const uint32_t v_sub = (((lane >> 3) & 1) << 3) + (lane & 7);
  const uint32_t v_chunk = 2 * warp + (lane >> 4);  // this warp's 16 output dims
  const uint32_t a_row = ((lane & 7) + 8 * ((lane >> 3) & 1));
  const uint32_t p_addr = smem_u32(pmat) + a_row * (kPRow * 2) + 16 * (lane >> 4);
  bool ok = true;
  float oacc[2][4];  // running P.V of rows gr / gr + 8, scaled to the running max
  zero4(oacc[0]);
  zero4(oacc[1]);
  float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;  // running max and sum
  float lse0 = -INFINITY, lse1 = -INFINITY;

  if (rounds > 0) {  // CTA-uniform: the piece holds keys of this query
    // R(-b w_f) and R(-(b + 2048) w_f), one per thread
    if (tid < 128) {
      float cs, sn;
      rope_cos_sin(-(bq + kWindow * (tid >> 6)), turns[tid & 63], cs, sn);
      ang[tid] = make_float2(cs, sn);
    }
    consumers_sync();
  }
  // Early start: round 0's keys rotated and split into B fragments before
  // the dependency wait, [k-step][hi x, lo x, hi y, lo y][fragment].
  uint32_t kfr[4][4][4];
  if (early) {
    if (rounds > 0) {
      const int32_t sb = s0 + key_in_round + gr;
      float2 kang[32];
#pragma unroll
      for (int sel = 0; sel < 2; ++sel) {
        const float2 *a = ang + ((sb + 8 * sel > bq) ? 64 : 0);
        const bool self = sb + 8 * sel == bq;  // offset 0: exactly the identity
#pragma unroll
        for (int f = 0; f < 16; ++f)
          kang[16 * sel + f] = self ? make_float2(1.f, 0.f) : cmul(tab[16 * sel + f], a[freq_of(f, tq)]);
      }
      const bool w = wait_round(0, &abort_flag);
      const bool okw = __all_sync(0xffffffffu, w) && !abort_flag;
      if (!okw && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
      ok = ok && okw;
      const uint32_t kbase = smem_base + th * kDecStageBytes;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t kx[4], ky[4];
        const uint32_t off = sw128(k_row, 2 * ks + k_chi);
        ldsm_x4(kbase + off, kx[0], kx[1], kx[2], kx[3]);
        ldsm_x4(kbase + 8192 + off, ky[0], ky[1], ky[2], ky[3]);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int j = 16 * (r >> 1) + 4 * ks + 2 * (r & 1);
          rot_split(kx[r], ky[r], kang[j], kang[j + 1], kfr[ks][0][r], kfr[ks][1][r], kfr[ks][2][r],
                    kfr[ks][3][r]);
        }
      }
    }
    pdl_wait();
    if (!overlap) pdl_launch_dependents();
    load_query();
  }
  if (bad && my_rank == 0 && g == 0 && tid == 0) set_err(p.err, MG_DERR_POSITION);
  for (int u = 0; u < rounds; ++u) {
    const int32_t r0 = s0 + u * kRound;  // first slot of the round
    const int32_t key0 = r0 + key_in_round;
    const int32_t sb = key0 + gr;
    const uint32_t kbase = smem_base + (u % kBufs) * kRoundSmem + th * kDecStageBytes;
    // the keys' offsets from the query: R(d) = R(s) R(-b) (s <= b) or
    // R(s) R(-b - 2048) (s > b), and R(0) = I exactly for the query's own slot
    float2 kang[32];
    if (!early) {
#pragma unroll
      for (int sel = 0; sel < 2; ++sel) {
        const float2 *a = ang + ((sb + 8 * sel > bq) ? 64 : 0);
        const bool self = sb + 8 * sel == bq;  // offset 0: exactly the identity
#pragma unroll
        for (int f = 0; f < 16; ++f)
          kang[16 * sel + f] = self ? make_float2(1.f, 0.f) : cmul(tab[16 * sel + f], a[freq_of(f, tq)]);
      }
      const bool w = wait_round(u, &abort_flag);
      const bool okw = __all_sync(0xffffffffu, w) && !abort_flag;
      if (!okw && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
      ok = ok && okw;
    }
    // the new token's row replaces the ring row of its slot: lane c writes
    // 16-byte chunk c of K (c < 16) or of V, and decode also stores it in the ring
    const bool patch_here = patch_mode && !bad && bq >= key0 && bq < key0 + 16;
    if (early && patch_here && ok) {
      // The keys are already rotated: the new key sits at offset 0 from the
      // query (no rotation), so the fragments of its row take k_new as the
      // hi part and zero as the lo part; its V row goes into shared memory
      // (read by P.V after the softmax barriers).
      const int rr = bq - key0;  // row among the warp's 16 keys: gr + 8 sel
      const bool mine = gr == (rr & 7);
      uint32_t nx[4][2], ny[4][2];  // the new key's dims 16 ks + 8 h8 + 2 tq (+ 64)
      const __nv_bfloat16 *kn = p.k_new + new_src;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int d = 16 * ks + 8 * h8 + 2 * tq;
          nx[ks][h8] = mine ? __ldg(reinterpret_cast<const unsigned int *>(kn + d)) : 0u;
          ny[ks][h8] = mine ? __ldg(reinterpret_cast<const unsigned int *>(kn + 64 + d)) : 0u;
        }
#pragma unroll
      for (int sel = 0; sel < 2; ++sel) {
        const bool hit = mine && sel == (rr >> 3);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            uint32_t(&f)[4][4] = kfr[ks];
            f[0][2 * sel + h8] = hit ? nx[ks][h8] : f[0][2 * sel + h8];
            f[1][2 * sel + h8] = hit ? 0u : f[1][2 * sel + h8];
            f[2][2 * sel + h8] = hit ? ny[ks][h8] : f[2][2 * sel + h8];
            f[3][2 * sel + h8] = hit ? 0u : f[3][2 * sel + h8];
          }
      }
      const uint32_t r = static_cast<uint32_t>(bq - r0 - th * kDecTile);
      const int c = lane & 15;
      if (lane >= 16) {
        const uint32_t addr = kbase + 16384 + (c >> 3) * 8192 + sw128(r, c & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(new_row.x),
                     "r"(new_row.y), "r"(new_row.z), "r"(new_row.w)
                     : "memory");
      }
      if (p.write_new) {
        const size_t dst = (static_cast<size_t>(head) * kWindow + bq) * kD;
        reinterpret_cast<uint4 *>((lane < 16 ? p.k_cache : p.v_cache) + dst)[c] = new_row;
      }
      __syncwarp();
    }
    if (!early && patch_here && ok) {
      const uint32_t r = static_cast<uint32_t>(bq - r0 - th * kDecTile);
      const int c = lane & 15;
      const uint32_t addr = kbase + (lane < 16 ? 0 : 16384) + (c >> 3) * 8192 + sw128(r, c & 7);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(new_row.x),
                   "r"(new_row.y), "r"(new_row.z), "r"(new_row.w)
                   : "memory");
      if (p.write_new) {
        const size_t dst = (static_cast<size_t>(head) * kWindow + bq) * kD;
        reinterpret_cast<uint4 *>((lane < 16 ? p.k_cache : p.v_cache) + dst)[c] = new_row;
      }
      __syncwarp();
    }
    // On a timeout the warp still runs every step below (shared-memory reads
    // only, so it stays in bounds) to keep the named barriers matched, and
    // drops its result.

    // ---------------------------------------------------- S = Q K'^T ----
    float sacc[2][4];  // [n8 tile][fragment]
    {
      float acc[2][4];
      zero4(acc[0]);
      zero4(acc[1]);
      if (early) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_16816(acc[0], qf[ks], kfr[ks][0][0], kfr[ks][0][1]);
          mma_16816(acc[1], qf[ks], kfr[ks][0][2], kfr[ks][0][3]);
          mma_16816(acc[0], qf[ks + 4], kfr[ks][2][0], kfr[ks][2][1]);
          mma_16816(acc[1], qf[ks + 4], kfr[ks][2][2], kfr[ks][2][3]);
          mma_16816(acc[0], qf[ks], kfr[ks][1][0], kfr[ks][1][1]);
          mma_16816(acc[1], qf[ks], kfr[ks][1][2], kfr[ks][1][3]);
          mma_16816(acc[0], qf[ks + 4], kfr[ks][3][0], kfr[ks][3][1]);
          mma_16816(acc[1], qf[ks + 4], kfr[ks][3][2], kfr[ks][3][3]);
        }
      } else
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t kx[4], ky[4];  // dims 16 ks.. and 64 + 16 ks..
        const uint32_t off = sw128(k_row, 2 * ks + k_chi);
        ldsm_x4(kbase + off, kx[0], kx[1], kx[2], kx[3]);
        ldsm_x4(kbase + 8192 + off, ky[0], ky[1], ky[2], ky[3]);
        uint32_t xh[4], xl[4], yh[4], yl[4];
#pragma unroll
        for (int sel = 0; sel < 2; ++sel)
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            const int r = 2 * sel + h8, j = 16 * sel + 4 * ks + 2 * h8;
            rot_split(kx[r], ky[r], kang[j], kang[j + 1], xh[r], xl[r], yh[r], yl[r]);
          }
        mma_16816(acc[0], qf[ks], xh[0], xh[1]);
        mma_16816(acc[1], qf[ks], xh[2], xh[3]);
        mma_16816(acc[0], qf[ks + 4], yh[0], yh[1]);
        mma_16816(acc[1], qf[ks + 4], yh[2], yh[3]);
        mma_16816(acc[0], qf[ks], xl[0], xl[1]);
        mma_16816(acc[1], qf[ks], xl[2], xl[3]);
        mma_16816(acc[0], qf[ks + 4], yl[0], yl[1]);
        mma_16816(acc[1], qf[ks + 4], yl[2], yl[3]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int32_t key = key0 + 8 * j + 2 * tq + (e & 1);
          sacc[j][e] = key < n_slots ? acc[j][e] * p.scale_log2 : -INFINITY;
        }
    }

    // -------------------------------------------------------- softmax ----
    float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
    float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (tq == 0) {
      red_m[warp * kGroup + gr] = mx0;
      red_m[warp * kGroup + gr + 8] = mx1;
    }
    consumers_sync();
    float Mn0 = M0, Mn1 = M1;  // the running max after this round
#pragma unroll
    for (int w = 0; w < kLocWarps; ++w) {
      Mn0 = fmaxf(Mn0, red_m[w * kGroup + gr]);
      Mn1 = fmaxf(Mn1, red_m[w * kGroup + gr + 8]);
    }
    const float Ms0 = Mn0 == -INFINITY ? 0.f : Mn0, Ms1 = Mn1 == -INFINITY ? 0.f : Mn1;
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float e0 = fast_exp2(sacc[j][0] - Ms0), e1 = fast_exp2(sacc[j][1] - Ms0);
      const float e2 = fast_exp2(sacc[j][2] - Ms1), e3 = fast_exp2(sacc[j][3] - Ms1);
      l0 += e0 + e1;
      l1 += e2 + e3;
      // key column in P: the slot's offset in the round
      const int kc = key_in_round + 8 * j + 2 * tq;
      pmat[gr * (kPRow / 2) + kc / 2] = pack_bf16x2(e0, e1);
      pmat[(gr + 8) * (kPRow / 2) + kc / 2] = pack_bf16x2(e2, e3);
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
    // rescale what earlier rounds accumulated to the new running max
    const float a0 = M0 == -INFINITY ? 0.f : fast_exp2(M0 - Ms0);
    const float a1 = M1 == -INFINITY ? 0.f : fast_exp2(M1 - Ms1);
    M0 = Mn0;
    M1 = Mn1;
    L0 *= a0;
    L1 *= a1;
#pragma unroll
    for (int w = 0; w < kLocWarps; ++w) {
      L0 += red_l[w * kGroup + gr];
      L1 += red_l[w * kGroup + gr + 8];
    }
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      oacc[n][0] *= a0;
      oacc[n][1] *= a0;
      oacc[n][2] *= a1;
      oacc[n][3] *= a1;
    }
    // --------------------------------- O[:, 16 w .. 16 w + 16) += P V ----
    {
      float pacc[2][2][4];  // [k-step parity][n8 tile]
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        zero4(pacc[v][0]);
        zero4(pacc[v][1]);
      }
      constexpr int kKk = kRound / 16;  // k-steps over the round's keys
      const uint32_t vround = smem_base + (u % kBufs) * kRoundSmem;
      uint32_t pa[kKk][4], vb[kKk][4];
#pragma unroll
      for (int kk = 0; kk < kKk; ++kk) {
        ldsm_x4(p_addr + kk * 32, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]);
        ldsm_x4_t(vround + (kk >> 2) * kDecStageBytes + 16384 + (v_chunk >> 3) * 8192 +
                      sw128(16 * (kk & 3) + v_sub, v_chunk & 7),
                  vb[kk][0], vb[kk][1], vb[kk][2], vb[kk][3]);
      }
#pragma unroll
      for (int kk = 0; kk < kKk; ++kk) {
        mma_16816(pacc[kk & 1][0], pa[kk], vb[kk][0], vb[kk][1]);
        mma_16816(pacc[kk & 1][1], pa[kk], vb[kk][2], vb[kk][3]);
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[n][e] += pacc[0][n][e] + pacc[1][n][e];
    }
    if (kRounds > 1) {
      // every warp is past its reads of this round's buffer and of P
      consumers_sync();
      if (tid == 0 && ok && u + kBufs < rounds) {
        issue_round(u + kBufs);
        ++issued;
      }
#pragma unroll
      for (int f = 0; f < 32; ++f) tab[f] = cmul(tab[f], step_round[freq_of(f & 15, tq)]);
    }
  }
  // Never leave the CTA with copies in flight: wait (full limit, no abort)
  // for the last round issued into each buffer -- a round without keys, or
  // one the loop gave up on after a timeout; a round already waited for
  // passes at once.
  if (tid == 0)
    for (int u = issued - 1; u >= 0 && u >= issued - kBufs; --u)
      if (!wait_round(u, nullptr)) set_err(p.err, MG_DERR_TIMEOUT);
  if (rounds > 0 && ok && L0 > 0.f && L1 > 0.f) {
    const float i0f = 1.f / L0, i1f = 1.f / L1;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      oacc[n][0] *= i0f;
      oacc[n][1] *= i0f;
      oacc[n][2] *= i1f;
      oacc[n][3] *= i1f;
    }
    lse0 = M0 + __log2f(L0);
    lse1 = M1 + __log2f(L1);
  } else {
    zero4(oacc[0]);
    zero4(oacc[1]);
  }

  // -------------- push this CTA's partial rows to the CTAs that own them ----
  // Head h belongs to CTA h / kOwned, which keeps it at inbox row
  // (h % kOwned) * kCl + source.
  __syncwarp();
  cluster_wait();  // every CTA of the cluster runs, its inbox barrier is set
  {
    const uint32_t inbox_s = smem_u32(inbox);
    const uint32_t own0 = gr / kOwned, own1 = (gr + 8) / kOwned;
    const uint32_t row0 = (gr % kOwned) * kCl + my_rank, row1 = ((gr + 8) % kOwned) * kCl + my_rank;
    const uint32_t bar0 = map_to_rank(bar_inbox, own0), bar1 = map_to_rank(bar_inbox, own1);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int d = 16 * warp + 8 * n + 2 * tq;
      st_async_f32x2(map_to_rank(inbox_s + 4 * (row0 * kD + d), own0), oacc[n][0], oacc[n][1], bar0);
      st_async_f32x2(map_to_rank(inbox_s + 4 * (row1 * kD + d), own1), oacc[n][2], oacc[n][3], bar1);
    }
    if (warp == 0 && tq == 0) {
      const uint32_t lse_s = inbox_s + 4 * (kOwned * kCl * kD);
      st_async_f32(map_to_rank(lse_s + 4 * row0, own0), lse0, bar0);
      st_async_f32(map_to_rank(lse_s + 4 * row1, own1), lse1, bar1);
    }
  }

  // ---------- merge the rows this CTA owns (heads kOwned * rank + j) ----
  // Every push into this CTA has landed once its inbox barrier completes;
  // the CTA reads and writes no other CTA's memory after its own pushes.
  const bool all_in = mbar_wait_cluster(bar_inbox, 0);
  if (!all_in && tid == 0) set_err(p.err, MG_DERR_TIMEOUT);
  if (all_in) {
    for (int i = tid; i < kOwned * kD; i += kLocThreads) {
      const int j = i / kD, d = i % kD;
      const float *rows = inbox + j * kCl * kD;
      const float *lse = inbox + kOwned * kCl * kD + j * kCl;
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kCl; ++c) M = fmaxf(M, lse[c]);
      float acc = 0.f, den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < kCl; ++c) {
          const float w = lse[c] == -INFINITY ? 0.f : fast_exp2(lse[c] - M);
          den += w;
          acc = fmaf(w, rows[c * kD + d], acc);
        }
      }
      const size_t orow = static_cast<size_t>(b) * kHq + g * kGroup + my_rank * kOwned + j;
      p.o[orow * kD + d] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
    }
  }
}

namespace {

template <int kRounds>
cudaError_t launch_local_rounds(const LocalParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                cudaStream_t s, int kernel_id) {
  using Plan = LocPlan<kRounds>;
  static_assert(Plan::kSmem <= 227 * 1024, "shared memory");
  static_assert(kGroup % Plan::kCl == 0, "the cluster's CTAs share the group's heads evenly");
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(local_attn_kernel<kRounds>),
                                   Plan::kSmem, kernel_id);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Plan::kCl, kHkv, p.batch);
  cfg.blockDim = dim3(kLocThreads);
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
  return cudaLaunchKernelEx(&cfg, local_attn_kernel<kRounds>, p, tk, tv);
}

}  // namespace

cudaError_t launch_local_attn(LocalParams p, const CUtensorMap &tk, const CUtensorMap &tv,
                              cudaStream_t s) {
  static_assert(kGroup == kLocCluster, "a 16-CTA cluster gives each CTA one head to merge");
  if (p.n != 1 || p.batch < 1) return cudaErrorInvalidValue;
  // One cluster per (sequence, KV head).  On this B300 at most 7 clusters of
  // 16 CTAs run at once (one per GPC), 15 of 8, 33 of 4: the fewest rounds
  // per CTA that put every pair in one wave.
  const int pairs = p.batch * kHkv;
  // The early start pays only while this kernel's clusters can be resident
  // beside the previous kernel's (two sets of 16-CTA clusters in 7 GPCs):
  // otherwise the late clusters would read the query after their keys
  // instead of beside them.
  if (pairs > 3) p.early = p.overlap = 0;
  if (pairs <= 7) return launch_local_rounds<1>(p, tk, tv, s, 2);
  if (pairs <= 15) return launch_local_rounds<2>(p, tk, tv, s, 7);
  return launch_local_rounds<4>(p, tk, tv, s, 8);
}

}  // namespace mg
