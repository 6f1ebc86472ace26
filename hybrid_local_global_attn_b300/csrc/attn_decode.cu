// attn_decode.cu -- split-KV flash-decode for one query token per sequence.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// section 01; "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
// section "长上下文仍然带来计算开销"): for the query at position p, softmax
// attention over the keys in [max(0, p-2047), p] with RoPE (local layer) or
// over [0, p] without RoPE (global layer); 16 query heads share one KV head.
//
// Design (HBM-bound: every K/V byte is read once):
//  * One CTA per (split, KV head, sequence).  It walks its share of the cache
//    in slot order -- the softmax does not care about key order, so a local
//    ring is read as the contiguous block of its 2048 slots and each slot's
//    position is recovered as p - ((p - slot) mod 2048).
//  * A producer warp streams 64-key K and V tiles with TMA (128-byte
//    swizzle, two 64-dim boxes per tile) into an mbarrier ring.
//  * Four consumer warps take 16 keys each of every tile.  The 16 query heads
//    of the KV group form the M = 16 side of mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate) for both Q.K^T and P.V; the K fragments are loaded
//    with ldmatrix and, in a local layer, rotated in registers (dimension i
//    and i+64 land in the same thread) with angles computed into shared
//    memory while the tiles are still in flight.  Online softmax in base 2
//    with quad shuffles; row sums stay per thread until the end.
//  * The four warps merge in shared memory into the CTA's partial (o / l,
//    lse).  Global layers (many splits) write it to the workspace and a
//    combine kernel merges the splits.  Local layers run the 16 splits of a
//    KV head as one thread-block cluster and merge through distributed
//    shared memory, writing the output directly.
//  * Optionally the token's own K/V is appended by the CTA that reads its
//    slot, before that tile is loaded (mg_append_decode).
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled
// box whose rows are 128 bytes.
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// Rotate the packed bf16 pairs (lo = dims i,i+1; hi = dims i+64,i+65) by the
// angles of frequencies i and i+1, in fp32, rounding back to bf16.
__device__ __forceinline__ void rot_pair(uint32_t &lo, uint32_t &hi, float c0, float s0, float c1,
                                         float s1) {
  const float x0 = bf16lo(lo), x1 = bf16hi(lo);
  const float y0 = bf16lo(hi), y1 = bf16hi(hi);
  lo = pack_bf16x2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
  hi = pack_bf16x2(x0 * s0 + y0 * c0, x1 * s1 + y1 * c1);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Compile-time configuration of the two decode variants.
template <bool kLocal>
struct DecCfg {
  // local: 16 CTAs x 128 keys cover the 2048-slot ring, one cluster per head
  static constexpr int kStages = kLocal ? 2 : 3;
  static constexpr int kCluster = kLocal ? 16 : 1;
  static constexpr int kMinBlocks = kLocal ? 1 : 2;
  static constexpr int kStageBytes = kDecStageBytes;
  static constexpr int kTableBytes = kLocal ? kStages * 32 * 128 * 8 : 0;  // float2 per entry
  // rows this CTA receives from every CTA of its cluster: o [rows][cluster][128], lse after
  static constexpr int kInboxBytes =
      kCluster > 1 ? ((kGroup * kD + kGroup) * 4 + 255) / 256 * 256 : 0;
  static constexpr int kRotBytes = kLocal ? 6 * 64 * 8 : 0;
  static constexpr int kSmem = kStages * kStageBytes + kTableBytes + kInboxBytes + kRotBytes +
                               1024 + 2 * 8 * kStages + 512;
};

}  // namespace

template <bool kLocal>
__global__ void __launch_bounds__(kDecThreads, DecCfg<kLocal>::kMinBlocks)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  using Cfg = DecCfg<kLocal>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float2 *table = reinterpret_cast<float2 *>(smem + NS * Cfg::kStageBytes);  // local only
  float *inbox = reinterpret_cast<float *>(smem + NS * Cfg::kStageBytes + Cfg::kTableBytes);
  float2 *rot = reinterpret_cast<float2 *>(smem + NS * Cfg::kStageBytes + Cfg::kTableBytes +
                                           Cfg::kInboxBytes);  // [6][64], local only
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NS * Cfg::kStageBytes + Cfg::kTableBytes +
                                                Cfg::kInboxBytes + Cfg::kRotBytes);
  uint64_t *turns = bars + 2 * NS;  // 64 entries

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * NS;

  // Prologue that touches no memory written by earlier kernels: it overlaps
  // the previous kernel's tail under programmatic dependent launch.
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kDecWarps);
    }
    fence_mbar_init();
  }
  if (kLocal) {
    if (threadIdx.x < 64) turns[threadIdx.x] = p.rope.turn[threadIdx.x];
    for (int i = threadIdx.x; i < 6 * 64; i += blockDim.x) rot[i] = p.rope.step[i / 64][i % 64];
  }
  if (warp == kDecWarps && lane == 0) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    // Warm L2 with the first tiles this CTA will stream while the previous
    // kernel is still running.  The range is what the split gets when the
    // query sits at max_len - 1 (local: fixed 128-slot pieces); only a
    // prefetch -- the loads that feed the math come after pdl_wait().
    int32_t c = kLocal ? kWindow / kDecLocalSplits : (p.max_len + p.splits - 1) / p.splits;
    c = (c + kDecTile - 1) / kDecTile * kDecTile;
    const int32_t first = split * c;
    const int32_t upto = min(min(first + (kLocal ? c : kDecPrefetchTiles * kDecTile), first + c),
                             kLocal ? p.slots : min(p.max_len, p.slots));
    for (int32_t row = first; row < upto; row += kDecTile)
      for (int x = 0; x < 2; ++x) {
        tma_prefetch_l2_3d(&tk, 64 * x, row, b * kHkv + g);
        tma_prefetch_l2_3d(&tv, 64 * x, row, b * kHkv + g);
      }
  }
  __syncthreads();
  // First half of a cluster barrier whose wait (before the first store into
  // another CTA's shared memory) proves every CTA of the cluster is running.
  if (Cfg::kCluster > 1) cluster_arrive_relaxed();
  pdl_wait();
  pdl_launch_dependents();

  // Local layers split the 2048-slot ring into fixed 128-slot pieces, so the
  // producer can start both tile loads before the query position is known.
  constexpr int kLocalChunk = kWindow / kDecLocalSplits;
  static_assert(!kLocal || kLocalChunk == NS * kDecTile, "a local CTA holds all its tiles");
  if (kLocal && warp == kDecWarps && lane == 0) {
    for (int t = 0; t < NS; ++t) {
      const uint32_t dst = smem_base + t * Cfg::kStageBytes;
      const uint32_t fb = bar_full + 8 * t;
      const int32_t row = split * kLocalChunk + t * kDecTile;
      mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
      tma_load_3d(dst, &tk, fb, 0, row, b * kHkv + g);
      tma_load_3d(dst + 8192, &tk, fb, 64, row, b * kHkv + g);
      tma_load_3d(dst + 16384, &tv, fb, 0, row, b * kHkv + g);
      tma_load_3d(dst + 24576, &tv, fb, 64, row, b * kHkv + g);
    }
  }

  const int32_t pq = p.pos[b];
  const bool bad = pq < 0 || pq >= p.max_len || (!kLocal && pq >= p.slots);
  int32_t n_slots = 0;
  if (!bad) n_slots = kLocal ? min(pq + 1, p.slots) : pq + 1;
  int32_t chunk = kLocalChunk;
  if (!kLocal) {
    chunk = (n_slots + p.splits - 1) / p.splits;
    chunk = (chunk + kDecTile - 1) / kDecTile * kDecTile;
  }
  const int32_t s0 = split * chunk;
  const int32_t s1 = min(s0 + chunk, n_slots);
  const bool empty = bad || s0 >= s1;
  const int ntiles = empty ? 0 : (s1 - s0 + kDecTile - 1) / kDecTile;
  const size_t row0 = static_cast<size_t>(b) * kHq + g * kGroup;  // first query row of the group
  if (bad && split == 0 && threadIdx.x == 0) set_err(p.err, MG_DERR_POSITION);

  // Where this CTA's partial of row r (o already divided by its softmax sum,
  // and lse) goes: the split-partial workspace, or -- in a cluster -- slot
  // `rank` of the inbox of the CTA that owns row r.
  constexpr int kOwnRows = kGroup / Cfg::kCluster;
  const uint32_t my_rank = Cfg::kCluster > 1 ? cluster_rank() : 0;
  const uint32_t inbox_s = smem_u32(inbox);
  auto emit_o = [&](int r, int d, float v) {
    if (Cfg::kCluster == 1) {
      p.part_o[((row0 + r) * p.splits + split) * kD + d] = v;
    } else {
      const int slot = (r % kOwnRows) * Cfg::kCluster + my_rank;
      st_cluster_f32(map_to_rank(inbox_s + 4 * (slot * kD + d), r / kOwnRows), v);
    }
  };
  auto emit_lse = [&](int r, float v) {
    if (Cfg::kCluster == 1) {
      p.part_lse[(row0 + r) * p.splits + split] = v;
    } else {
      const int slot = (r % kOwnRows) * Cfg::kCluster + my_rank;
      st_cluster_f32(map_to_rank(inbox_s + 4 * (kGroup * kD + slot), r / kOwnRows), v);
    }
  };

  const int32_t my_slot = kLocal ? pq % kWindow : pq;  // slot of the query token
  const bool fused_here = p.k_new != nullptr && !empty && my_slot >= s0 && my_slot < s1;
  bool ok = true;
  if (kLocal && warp == kDecWarps) {
    // Fused append (local): write the token's row into the cache.  This CTA's
    // own copy of the slot was loaded before the write may have landed; the
    // consumer warp that owns the row patches it in shared memory instead.
    if (fused_here) {
      const size_t src = (static_cast<size_t>(b) * kHkv + g) * kD;
      const size_t dst = ((static_cast<size_t>(b) * kHkv + g) * p.slots + my_slot) * kD;
      const int c = lane & 15;
      if (lane < 16)
        reinterpret_cast<uint4 *>(p.k_cache + dst)[c] =
            __ldg(reinterpret_cast<const uint4 *>(p.k_new + src) + c);
      else
        reinterpret_cast<uint4 *>(p.v_cache + dst)[c] =
            __ldg(reinterpret_cast<const uint4 *>(p.v_new + src) + c);
    }
    if (lane == 0) {  // never leave the CTA with copies in flight
      for (int t = 0; t < NS; ++t) (void)mbar_wait(bar_full + 8 * t, 0, nullptr);
    }
    __syncwarp();
  } else if (warp == kDecWarps) {
    // ------------------------------------------------ TMA producer warp ----
    if (!empty) {
      // Fused append (global): the query token's K/V row lands in its slot
      // before the tile that holds the slot is read (the TMA read goes
      // through the async proxy, hence the proxy fence after the stores).
      if (fused_here) {
        const size_t src = (static_cast<size_t>(b) * kHkv + g) * kD;
        const size_t dst = ((static_cast<size_t>(b) * kHkv + g) * p.slots + my_slot) * kD;
        const int c = lane & 15;
        if (lane < 16)
          reinterpret_cast<uint4 *>(p.k_cache + dst)[c] =
              __ldg(reinterpret_cast<const uint4 *>(p.k_new + src) + c);
        else
          reinterpret_cast<uint4 *>(p.v_cache + dst)[c] =
              __ldg(reinterpret_cast<const uint4 *>(p.v_new + src) + c);
        fence_proxy_async_global();
        __syncwarp();
      }
      if (lane == 0) {
        const int32_t c2 = b * kHkv + g;
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
          const int st = t % NS;
          if (t >= NS && !mbar_wait(bar_empty + 8 * st, ((t / NS) - 1) & 1, &abort_flag)) {
            abort_flag = 1;
            set_err(p.err, MG_DERR_TIMEOUT);
            break;
          }
          const uint32_t dst = smem_base + st * Cfg::kStageBytes;
          const uint32_t fb = bar_full + 8 * st;
          const int32_t row = s0 + t * kDecTile;
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          tma_load_3d(dst, &tk, fb, 0, row, c2);
          tma_load_3d(dst + 8192, &tk, fb, 64, row, c2);
          tma_load_3d(dst + 16384, &tv, fb, 0, row, c2);
          tma_load_3d(dst + 24576, &tv, fb, 64, row, c2);
          ++issued;
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the
        // last stages issued.
        for (int t = max(0, issued - NS); t < issued; ++t)
          (void)mbar_wait(bar_full + 8 * (t % NS), (t / NS) & 1, nullptr);
      }
      __syncwarp();
    }
  } else if (!empty) {
    // ------------------------------------------------------ consumer warps ----
    const int gr = lane >> 2;  // fragment row group (0..7)
    const int tq = lane & 3;   // thread in quad
    const int tid = threadIdx.x;

    // Q fragments (A operand, 16 heads x 128 dims): loads issued first so
    // their latency overlaps the angle computation below.
    uint32_t qf[8][4];
    {
      const __nv_bfloat16 *q0 = p.q + (row0 + gr) * kD;
      const __nv_bfloat16 *q1 = q0 + 8 * kD;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c = ks * 16 + 2 * tq;
        qf[ks][0] = __ldg(reinterpret_cast<const unsigned int *>(q0 + c));
        qf[ks][1] = __ldg(reinterpret_cast<const unsigned int *>(q1 + c));
        qf[ks][2] = __ldg(reinterpret_cast<const unsigned int *>(q0 + c + 8));
        qf[ks][3] = __ldg(reinterpret_cast<const unsigned int *>(q1 + c + 8));
      }
    }
    if (kLocal) {
      // This thread's 16 frequencies: i = 16 ks + 2 tq + 8 h8 + e, entry
      // f = 4 ks + 2 h8 + e.  Held in registers (the table stores below
      // would otherwise force a reload of each one).
      uint64_t tr[16];
#pragma unroll
      for (int f = 0; f < 16; ++f) tr[f] = turns[(f >> 2) * 16 + 2 * tq + 8 * ((f >> 1) & 1) + (f & 1)];
      // Angles of this thread's keys (2 per tile), computed while the tiles
      // are in flight; table entry j = 16 * key_sel + f.  Only the first key
      // is evaluated directly; the others sit 8, 64 or 72 slots further on,
      // i.e. 8, 64 or 72 positions (minus 2048 across the ring's wrap point),
      // and are obtained by multiplying with that step's rotation.
      {
        const int32_t sb = s0 + warp * 16 + gr;
        const int32_t kb = pq - ((pq - sb) & (kWindow - 1));
        float2 base[16];
#pragma unroll
        for (int f = 0; f < 16; ++f) rope_cos_sin(kb, tr[f], base[f].x, base[f].y);
#pragma unroll
        for (int f = 0; f < 16; ++f) table[f * 128 + tid] = base[f];
        const int nk = 2 * min(ntiles, NS);
        for (int k = 1; k < nk; ++k) {
          const int t = k >> 1, sel = k & 1;
          const int32_t delta = 64 * t + 8 * sel;
          const int32_t kd = pq - ((pq - (sb + delta)) & (kWindow - 1));
          const int ridx = (delta == 8 ? 0 : (delta == 64 ? 1 : 2)) + (kd - kb != delta ? 3 : 0);
          float2 r[16];  // all loads first: the table stores below would serialize them
#pragma unroll
          for (int f = 0; f < 16; ++f)
            r[f] = rot[ridx * 64 + (f >> 2) * 16 + 2 * tq + 8 * ((f >> 1) & 1) + (f & 1)];
#pragma unroll
          for (int f = 0; f < 16; ++f)
            table[(t * 32 + 16 * sel + f) * 128 + tid] = make_float2(
                base[f].x * r[f].x - base[f].y * r[f].y, base[f].y * r[f].x + base[f].x * r[f].y);
        }
      }
      // rotate q by R(p)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {  // dims c..c+1 then c+8..c+9
          const int f = 4 * ks + 2 * h8;
          float c0, s0f, c1, s1f;
          rope_cos_sin(pq, tr[f], c0, s0f);
          rope_cos_sin(pq, tr[f + 1], c1, s1f);
          rot_pair(qf[ks][2 * h8], qf[ks + 4][2 * h8], c0, s0f, c1, s1f);
          rot_pair(qf[ks][2 * h8 + 1], qf[ks + 4][2 * h8 + 1], c0, s0f, c1, s1f);
        }
      }
    }

    float oacc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = p.scale_log2;

    // per-lane ldmatrix row/chunk selectors
    const uint32_t k_row = warp * 16 + ((lane >> 4) << 3) + (lane & 7);  // key row in tile
    const uint32_t k_chi = (lane >> 3) & 1;                               // +8 dims
    const uint32_t v_row = warp * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
    const uint32_t v_chi = lane >> 4;                                     // +8 dims

    for (int t = 0; t < ntiles; ++t) {
      const int st = t % NS;
      // ldmatrix / mma.sync are warp-collective: the whole warp goes on or stops
      if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (t / NS) & 1, &abort_flag))) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
        ok = false;
        break;
      }
      const int32_t key0 = s0 + t * kDecTile + warp * 16;  // slot of this warp's first key
      if (key0 < s1) {
        const uint32_t kbase = smem_base + st * Cfg::kStageBytes;
        const uint32_t vbase = kbase + 16384;
        if (kLocal && fused_here && my_slot >= key0 && my_slot < key0 + 16) {
          // the token's own K/V replace the row loaded for its slot: lane c
          // writes 16-byte chunk c of K (c < 16) or of V
          const uint32_t kr = static_cast<uint32_t>(my_slot - s0 - t * kDecTile);
          const int c = lane & 15;
          const size_t src = (static_cast<size_t>(b) * kHkv + g) * kD;
          const uint4 val = (lane < 16) ? __ldg(reinterpret_cast<const uint4 *>(p.k_new + src) + c)
                                        : __ldg(reinterpret_cast<const uint4 *>(p.v_new + src) + c);
          const uint32_t base = (lane < 16) ? kbase : vbase;
          const uint32_t addr = base + (c >> 3) * 8192 + sw128(kr, c & 7);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(val.x),
                       "r"(val.y), "r"(val.z), "r"(val.w)
                       : "memory");
          __syncwarp();
        }
        float sacc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t lo[4], hi[4];
          // dims 16ks.. (box 0) and 16ks+64.. (box 1): same row and chunk
          const uint32_t off = sw128(k_row, 2 * ks + k_chi);
          ldsm_x4(kbase + off, lo[0], lo[1], lo[2], lo[3]);
          ldsm_x4(kbase + 8192 + off, hi[0], hi[1], hi[2], hi[3]);
          if (kLocal) {
            const int tt = min(t, NS - 1);  // local CTAs hold at most NS tiles
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
#pragma unroll
              for (int sel = 0; sel < 2; ++sel) {
                const int j = 16 * sel + 4 * ks + 2 * h8;
                const float2 a = table[(tt * 32 + j) * 128 + tid];
                const float2 c = table[(tt * 32 + j + 1) * 128 + tid];
                rot_pair(lo[2 * sel + h8], hi[2 * sel + h8], a.x, a.y, c.x, c.y);
              }
            }
          }
          mma_16816(sacc[0], qf[ks], lo[0], lo[1]);
          mma_16816(sacc[1], qf[ks], lo[2], lo[3]);
          mma_16816(sacc[0], qf[ks + 4], hi[0], hi[1]);
          mma_16816(sacc[1], qf[ks + 4], hi[2], hi[3]);
        }

        // scale to the base-2 domain and mask keys past the split's end
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int32_t key = key0 + 8 * j + 2 * tq + (e & 1);
            sacc[j][e] = (key < s1) ? sacc[j][e] * sl2 : -INFINITY;
          }
        }
        float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
        float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: key0 < s1
        const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pr[j][0] = fast_exp2(sacc[j][0] - mn0);
          pr[j][1] = fast_exp2(sacc[j][1] - mn0);
          pr[j][2] = fast_exp2(sacc[j][2] - mn1);
          pr[j][3] = fast_exp2(sacc[j][3] - mn1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          oacc[i][0] *= a0;
          oacc[i][1] *= a0;
          oacc[i][2] *= a1;
          oacc[i][3] *= a1;
        }
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);

        // O += P V : V rows are keys; ldmatrix.trans gives the col-major B
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
          const uint32_t chunk16 = nd + v_chi;  // 16-byte chunk over the 128 dims
          const uint32_t addr = vbase + (chunk16 >> 3) * 8192 + sw128(v_row, chunk16 & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma_16816(oacc[nd], pa, b0, b1);
          mma_16816(oacc[nd + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // ------------------------------------------- merge the four warps ----
    // Each warp rescales its own accumulators by 2^(m_w - M) / L in
    // registers; the four scaled slices are then summed from shared memory.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    constexpr int kRowPad = kD + 8;  // padded row stride (floats) of the slices
    // A local CTA loaded all its tiles up front, including any past its last
    // key: those copies must have landed before the stage memory is reused.
    if (kLocal)
      for (int t = ntiles; t < NS; ++t) (void)mbar_wait(bar_full + 8 * t, 0, nullptr);
    // every consumer is past its last read of the tiles before the stage
    // memory is reused for the merge
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    float *mo = reinterpret_cast<float *>(smem);  // [4 warps][16 rows][kRowPad]
    float *ml = mo + kDecWarps * kGroup * kRowPad;  // [4][16] m, then [4][16] l
    if (tq == 0) {
      ml[warp * kGroup + gr] = ok ? m0 : -INFINITY;
      ml[warp * kGroup + gr + 8] = ok ? m1 : -INFINITY;
      ml[kDecWarps * kGroup + warp * kGroup + gr] = ok ? l0 : 0.f;
      ml[kDecWarps * kGroup + warp * kGroup + gr + 8] = ok ? l1 : 0.f;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    float Mr[2], Lr[2], f[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = gr + 8 * h;
      float mw[kDecWarps], M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        mw[w] = ml[w * kGroup + r];
        M = fmaxf(M, mw[w]);
      }
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w)
        L += (mw[w] == -INFINITY) ? 0.f
                                  : fast_exp2(mw[w] - M) * ml[kDecWarps * kGroup + w * kGroup + r];
      Mr[h] = M;
      Lr[h] = L;
      const float mine = mw[warp];
      f[h] = (L > 0.f && mine != -INFINITY) ? fast_exp2(mine - M) / L : 0.f;
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      const int c = nd * 8 + 2 * tq;
      *reinterpret_cast<float2 *>(&mo[(warp * kGroup + gr) * kRowPad + c]) =
          make_float2(oacc[nd][0] * f[0], oacc[nd][1] * f[0]);
      *reinterpret_cast<float2 *>(&mo[(warp * kGroup + gr + 8) * kRowPad + c]) =
          make_float2(oacc[nd][2] * f[1], oacc[nd][3] * f[1]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    // Sum the four scaled slices and send each row straight to where it is
    // merged next: the workspace (split partials of a global layer) or the
    // inbox of the cluster CTA that owns the row (local layer).
    if (Cfg::kCluster > 1) cluster_wait();  // every CTA of the cluster runs
#pragma unroll 4
    for (int i = tid; i < kGroup * kD; i += kDecWarps * 32) {
      const int r = i / kD, d = i % kD;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) acc += mo[(w * kGroup + r) * kRowPad + d];
      emit_o(r, d, acc);
    }
    if (warp == 0 && tq == 0) {
      emit_lse(gr, Lr[0] > 0.f ? Mr[0] + __log2f(Lr[0]) : -INFINITY);
      emit_lse(gr + 8, Lr[1] > 0.f ? Mr[1] + __log2f(Lr[1]) : -INFINITY);
    }
  } else {
    // no keys for this split: lse = -inf, o = 0 (a local CTA's tile copies
    // may still be landing in its stage memory, so they are waited for:
    // the CTA must not retire with copies in flight)
    if (kLocal && warp < kDecWarps)
      for (int t = 0; t < NS; ++t) (void)mbar_wait(bar_full + 8 * t, 0, nullptr);
    if (warp < kDecWarps) {
      if (Cfg::kCluster > 1) cluster_wait();
      for (int i = threadIdx.x; i < kGroup * kD; i += kDecWarps * 32) emit_o(i / kD, i % kD, 0.f);
      if (threadIdx.x < kGroup) emit_lse(threadIdx.x, -INFINITY);
    }
  }

  if (Cfg::kCluster > 1) {
    // the producer warp completes the first cluster barrier phase too
    if (warp == kDecWarps) cluster_wait();
    // ------------ merge the rows this CTA owns from its inbox, write o ----
    constexpr int kRowsPerRank = kGroup / Cfg::kCluster;
    cluster_sync_all();  // all pushes have landed; no remote access after this
    if (warp < kDecWarps) {
      const uint32_t rank = cluster_rank();
      const int d = threadIdx.x;  // 0..127
      for (int rr = 0; rr < kRowsPerRank; ++rr) {
        const int r = rank * kRowsPerRank + rr;
        const float *lse = inbox + kGroup * kD + rr * Cfg::kCluster;
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < Cfg::kCluster; ++j) M = fmaxf(M, lse[j]);
        float acc = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int j = 0; j < Cfg::kCluster; ++j) {
            const float w = lse[j] == -INFINITY ? 0.f : fast_exp2(lse[j] - M);
            den += w;
            acc = fmaf(w, inbox[(rr * Cfg::kCluster + j) * kD + d], acc);
          }
        }
        p.o[(row0 + r) * kD + d] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
      }
    }
  }
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t s) {
  if (p.kind == 0) {
    using Cfg = DecCfg<true>;
    static_assert(kGroup % Cfg::kCluster == 0, "rows split evenly over the cluster");
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(decode_kernel<true>),
                                     Cfg::kSmem, 2);
    if (e != cudaSuccess) return e;
    if (p.splits != Cfg::kCluster) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits, kHkv, p.batch);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = Cfg::kCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_kernel<true>, p, tk, tv);
  }
  using Cfg = DecCfg<false>;
  cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void *>(decode_kernel<false>), Cfg::kSmem, 0);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, kHkv, p.batch);
  return launch_pdl(decode_kernel<false>, grid, dim3(kDecThreads), Cfg::kSmem, s, p, tk, tv);
}

}  // namespace mg
