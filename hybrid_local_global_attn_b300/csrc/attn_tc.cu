// attn_tc.cu -- tensor-core (tcgen05 / TMEM) attention for a block of query
// tokens: speculative verify and causal chunked prefill.
//
// What it computes: the query at position q sees the cached keys before the
// block start c0 that fall in its key set, plus the block's own keys up to q
// (causal inside the block) -- the parallel verify pass of a 16-token draft
// ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？", section 04;
// "Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析", section
// "第三招") and chunked prompt processing, full attention that stays quadratic
// in global layers ("Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse
// Glimmer", section "长上下文仍然带来计算开销").  Key sets: [q-2047, q] with
// RoPE (local; operands pre-rotated by rope_stage) or [0, q] without RoPE
// (global, operands read straight from the cache and the block).
//
// Tiling: a CTA owns 8 consecutive query positions of one KV group: 8
// positions x 16 query heads form one M = 128 tile (rows r = 16 * position +
// head).  Key tiles hold 256 keys and are aligned to c0, so a tile never
// straddles the cache and the block.
//
// The issue cost of one tcgen05.mma barely depends on N (on this B300 an
// M128 N128 K16 takes ~119 cycles with both operands in shared memory, an
// M128 N256 K16 ~139), so the scores are computed 256 keys at a time: S =
// Q K^T is 8 M128 N256 K16 MMAs, O += P V 16 M128 N128 K16 MMAs with P
// from TMEM.  TMEM holds S (256 fp32 columns), P (256 keys as bf16 pairs,
// 128 columns) and O (128 columns); because P has its own columns, S of the
// next tile is computed as soon as the softmax has loaded S into registers,
// and P.V of a tile overlaps Q.K^T of the next.
//
// Warp roles (320 threads):
//   warps 0-3  softmax of keys 0..127 of every key tile (thread = row = lane)
//   warps 4-7  softmax of keys 128..255 of the same rows; the two halves
//              exchange their row maxima once per tile
//   warp 8     TMA producer (Q once; K in a 2-deep ring of 256-key tiles,
//              V in a 2-deep ring of 128-key half tiles)
//   warp 9     TMEM owner and single-thread MMA issuer
// Per key tile: S = Q K^T, softmax in registers with a lazily rescaled
// running max (rescale only when the max grows by more than 2^8), P to TMEM,
// O += P V (V as an MN-major operand).
// Splits (verify): the cache part is cut across CTAs, split s of S taking
// every S-th key tile (s, s + S, ...: the CTAs then stream neighbouring
// tiles at any moment); each writes (o/l, lse) and the combine kernel
// merges them.
//
// Local layers (operands staged by rope_stage, rotated by their absolute
// positions) run the precise form of the kernel: queries and keys arrive as
// bf16 pairs hi = bf16(x), lo = bf16(x - hi) of the fp32 rotation, and
// S = Qhi Khi^T + Qlo Khi^T + Qhi Klo^T (24 MMAs per key tile instead of 8)
// carries the rounding of the rotated operands at about 2^-17 of |q||k|
// instead of 2^-9 -- one bf16 rounding moves a score by ~0.04 when scaled
// scores spread by ~40, enough to shift a peaked softmax row by several
// 1e-2.  Shared memory then holds Qhi and Qlo (64 KB), one key tile's hi and
// lo halves (64 KB each, each released as soon as its MMAs have run) and V
// in a 2-deep ring of 64-key quarter tiles.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kTcKeys, 0, 0);
// Shared-memory plan per form: Q bytes (hi, then lo in the precise form) and
// the V stage (128-key halves, or 64-key quarters in the precise form); the
// two 64 KB key buffers are K stages (plain) or a tile's hi and lo (precise).
template <bool kPrecise> struct TcPlan {
  static constexpr int kQ = kPrecise ? 2 * kTcQBytes : kTcQBytes;
  static constexpr int kVRows = kPrecise ? kTcKeys / 4 : kTcVRows;  // keys per V stage
  static constexpr int kVParts = kTcKeys / kVRows;                    // V stages per key tile
  static constexpr int kVBytes = kVRows * kRowBytes;
  static constexpr int kSmem = kQ + 2 * kTcKTileBytes + kTcVStages * kVBytes + 1024 + 256;
};
static_assert(TcPlan<true>::kSmem <= kTcSmem && TcPlan<false>::kSmem <= kTcSmem, "shared memory");
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct TileInfo {
  int32_t c0, qa, qz;     // block start, first and last valid query position
  int32_t cbase;          // cache tiles end here: c0, or c0 rounded up to 256 (paged)
  int32_t ncache, nnew;   // tiles from the cache part / the block part
  int32_t u_begin, v_lo;  // first cache tile index (from cbase down), first block tile
  int32_t u_step;         // cache tile index step between a CTA's tiles (the split count)
};

__device__ __forceinline__ int32_t tile_kp0(const TileInfo &ti, int t) {
  if (t < ti.ncache) return ti.cbase - kTcKeys * (ti.u_begin + t * ti.u_step + 1);
  return ti.c0 + kTcKeys * (ti.v_lo + (t - ti.ncache));
}

}  // namespace

template <bool kPrecise>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tka, const __grid_constant__ CUtensorMap tva,
                   const __grid_constant__ CUtensorMap tkb,
                   const __grid_constant__ CUtensorMap tvb,
                   const __grid_constant__ CUtensorMap tql,
                   const __grid_constant__ CUtensorMap tkl) {
  using Plan = TcPlan<kPrecise>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_base_slot;
  __shared__ float red_x[2][kTcRows];  // per tile: the two halves' row maxima
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase;                              // Q (precise: hi, then lo)
  const uint32_t sK = sbase + Plan::kQ;                   // two 64 KB key buffers
  const uint32_t sV = sK + 2 * kTcKTileBytes;             // V ring: stage s at +kVBytes*s
  const uint32_t sBar = sV + kTcVStages * Plan::kVBytes;
  // barrier addresses
  const uint32_t bar_q = sBar;                             // Q landed
  const uint32_t bar_kf = sBar + 8;                        // [2] key buffer full
  const uint32_t bar_ke = bar_kf + 8 * kTcKStages;         // [2] key buffer free
  const uint32_t bar_vf = bar_ke + 8 * kTcKStages;         // [kTcVStages] V stage full
  const uint32_t bar_ve = bar_vf + 8 * kTcVStages;         // [kTcVStages] V stage free
  const uint32_t bar_s = bar_ve + 8 * kTcVStages;          // S ready
  const uint32_t bar_sfree = bar_s + 8;                    // S loaded by the softmax (256)
  const uint32_t bar_p = bar_sfree + 8;                    // P ready (256 arrivals)
  const uint32_t bar_pfree = bar_p + 8;                    // P.V retired: P and O free
  const uint32_t bar_done = bar_pfree + 8;                 // all MMAs retired

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int split = blockIdx.x % p.splits;
  const int qb = p.qblocks - 1 - static_cast<int>(blockIdx.x / p.splits);  // heavy blocks first
  const bool local = (p.kind == 0);

  pdl_wait();  // positions, block K/V and (local) staged operands come from earlier kernels
  pdl_launch_dependents();

  // ------------------------------------------------------ tile schedule ----
  TileInfo ti;
  ti.c0 = p.pos0[b];
  const bool bad = ti.c0 < 0 || static_cast<int64_t>(ti.c0) + p.n > p.max_len ||
                   (!p.staged && ti.c0 > p.slots);
  // A paged cache's tiles are aligned to 256 so that each lies in one page;
  // the top one then reaches past c0 and its keys >= c0 are masked.
  ti.cbase = (p.map.table != nullptr && !local) ? (ti.c0 + kTcKeys - 1) / kTcKeys * kTcKeys : ti.c0;
  ti.qa = ti.c0 + kTcPosPerCta * qb;
  ti.qz = min(ti.qa + kTcPosPerCta - 1, ti.c0 + p.n - 1);
  ti.ncache = ti.nnew = ti.u_begin = ti.v_lo = 0;
  ti.u_step = p.splits;
  if (!bad) {
    const int32_t lo = local ? max(0, ti.qa - p.window + 1) : 0;
    const int32_t U = ti.c0 > lo ? (ti.c0 - lo + kTcKeys - 1) / kTcKeys : 0;
    // split s takes the cache tiles s, s + S, s + 2S, ... (S splits)
    ti.u_begin = split;
    ti.ncache = split < U ? (U - split + p.splits - 1) / p.splits : 0;
    if (split == p.splits - 1) {
      ti.v_lo = local ? max(0, ti.qa - p.window + 1 - ti.c0) / kTcKeys : 0;
      const int32_t v_hi = (ti.qz - ti.c0) / kTcKeys;
      ti.nnew = v_hi - ti.v_lo + 1;
    }
  }
  const int ntiles = ti.ncache + ti.nnew;

  // The producer lane sets up the barriers and at once issues every copy the
  // first key tile needs (Q, K and both V halves of tile 0: no stage waits),
  // so they overlap the TMEM allocation and the CTA barrier below.
  // Cache tile t lies in rows [crow0, crow0 + 256) of outer index couter
  // (linear: rows from 0 of the sequence's head; paged: its page).  K of
  // tile t + 1 is issued before V of tile t, so two tiles' entries live.
  int32_t crow0[2] = {0, 0}, couter[2] = {b * kHkv + g, b * kHkv + g};
  auto locate = [&](int t) {
    if (p.map.table == nullptr || t >= ti.ncache) return;
    const int32_t kp0 = tile_kp0(ti, t);
    int32_t r, o;
    cache_coord(p.map, b, g, kp0, &r, &o, p.err);
    crow0[t & 1] = kp0 - r;
    couter[t & 1] = o;
  };
  // keys kp0.. (rows) of K or V into dst (two 64-dim boxes), completing on
  // fb; `lo`: the lo halves of staged keys (precise form)
  auto load = [&](bool is_v, int t, int32_t kp0, uint32_t dst, uint32_t bytes, uint32_t fb,
                  bool lo = false) {
    const CUtensorMap *ma = is_v ? &tva : (lo ? &tkl : &tka);
    const CUtensorMap *mb = is_v ? &tvb : &tkb;
    mbar_arrive_expect_tx(fb, bytes);
    for (int x = 0; x < 2; ++x) {
      const uint32_t d = dst + x * (bytes / 2);
      if (p.staged)
        tma_load_3d(d, ma, fb, 64 * x, kp0 - ti.c0 + kWindow, b * kHkv + g);
      else if (t < ti.ncache)
        tma_load_3d(d, ma, fb, 64 * x, kp0 - crow0[t & 1], couter[t & 1]);
      else
        tma_load_4d(d, mb, fb, 64 * x, g, kp0 - ti.c0, b);
    }
  };
  int issued_k = 0, issued_v = 0;
  int issued_part[2] = {0, 0};  // precise form: copies issued into each key buffer
  bool ok = true;
  // Plain form: K of tile t reuses the stage of tile t - 2 once its
  // S = Q K^T has run.  Precise form: the hi and lo halves of tile t go to
  // buffers 0 and 1, each once the MMAs of tile t - 1 that read it have run.
  auto load_k = [&](int t) -> bool {
    if (kPrecise) {
      for (int part = 0; part < 2; ++part) {
        if (t >= 1 && !mbar_wait(bar_ke + 8 * part, (t - 1) & 1, &abort_flag)) return false;
        load(false, t, tile_kp0(ti, t), sK + part * kTcKTileBytes, kTcKTileBytes,
             bar_kf + 8 * part, part == 1);
        ++issued_part[part];
      }
      ++issued_k;
      return true;
    }
    const int ks = t % kTcKStages;
    if (t >= kTcKStages &&
        !mbar_wait(bar_ke + 8 * ks, ((t / kTcKStages) - 1) & 1, &abort_flag))
      return false;
    locate(t);
    load(false, t, tile_kp0(ti, t), sK + ks * kTcKTileBytes, kTcKTileBytes, bar_kf + 8 * ks);
    ++issued_k;
    return true;
  };
  // K runs a tile ahead of V (S = Q K^T of tile t + 1 is issued before
  // P.V of tile t); V half u = 2 t + h reuses the stage of half u - 2
  // once its P.V has run
  if (warp == 8 && lane == 0) {
    abort_flag = 0;
    if (bad && split == 0 && qb == 0) set_err(p.err, MG_DERR_POSITION);
    mbar_init(bar_q, 1);
    for (int i = 0; i < kTcKStages; ++i) {
      mbar_init(bar_kf + 8 * i, 1);
      mbar_init(bar_ke + 8 * i, 1);
    }
    for (int i = 0; i < kTcVStages; ++i) {
      mbar_init(bar_vf + 8 * i, 1);
      mbar_init(bar_ve + 8 * i, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 256);
    mbar_init(bar_p, 256);
    mbar_init(bar_pfree, 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
    if (ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tka);
      tma_prefetch_desc(&tva);
      tma_prefetch_desc(&tkb);
      tma_prefetch_desc(&tvb);
      const int32_t q_t0 = kTcPosPerCta * qb;  // position index within the block
      mbar_arrive_expect_tx(bar_q, Plan::kQ);
      for (int x = 0; x < 2; ++x) {
        tma_load_4d(sQ + x * (kTcQBytes / 2), &tq, bar_q, 64 * x, kGroup * g, q_t0, b);
        if (kPrecise)
          tma_load_4d(sQ + kTcQBytes + x * (kTcQBytes / 2), &tql, bar_q, 64 * x, kGroup * g,
                      q_t0, b);
      }
      (void)load_k(0);  // first use of the key buffers: no wait
      for (int h = 0; h < kTcVStages; ++h) {  // V stages 0 and 1 of tile 0: no wait
        load(true, 0, tile_kp0(ti, 0) + Plan::kVRows * h, sV + h * Plan::kVBytes, Plan::kVBytes,
             bar_vf + 8 * h);
        ++issued_v;
      }
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&tmem_base_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_slot;
  constexpr uint32_t kColP = kTcKeys, kColO = kTcKeys + kTcKeys / 2;  // S at 0

  if (warp == 8) {
    // ------------------------------------------------------- producer ----
    if (lane == 0 && ntiles > 0) {
      // K(0) and the first V stages of tile 0 went out before the CTA barrier
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles && !load_k(t + 1)) {
          ok = false;
          break;
        }
        for (int h = 0; h < Plan::kVParts; ++h) {
          const int u = Plan::kVParts * t + h, vs = u % kTcVStages;
          if (u < kTcVStages) continue;  // issued already
          if (!mbar_wait(bar_ve + 8 * vs, ((u / kTcVStages) - 1) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          load(true, t, tile_kp0(ti, t) + Plan::kVRows * h, sV + vs * Plan::kVBytes,
               Plan::kVBytes, bar_vf + 8 * vs);
          ++issued_v;
        }
      }
      if (!ok) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
      }
      // no copies may be in flight when the CTA retires
      (void)mbar_wait(bar_q, 0, nullptr);
      if (kPrecise) {
        for (int part = 0; part < 2; ++part)
          if (issued_part[part] > 0)
            (void)mbar_wait(bar_kf + 8 * part, (issued_part[part] - 1) & 1, nullptr);
      } else {
        for (int t = max(0, issued_k - kTcKStages); t < issued_k; ++t)
          (void)mbar_wait(bar_kf + 8 * (t % kTcKStages), (t / kTcKStages) & 1, nullptr);
      }
      for (int u = max(0, issued_v - kTcVStages); u < issued_v; ++u)
        (void)mbar_wait(bar_vf + 8 * (u % kTcVStages), (u / kTcVStages) & 1, nullptr);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(bar_q, 0, &abort_flag);
      // S = Q K(t)^T
      auto qk = [&](int t) -> bool {
        const int st = t % kTcKStages;
        if (!mbar_wait(bar_kf + 8 * st, (t / kTcKStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t ks = sK + st * kTcKTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_ss(tbase, smem_desc_sw128(sQ + (kk >> 2) * (kTcQBytes / 2) + (kk & 3) * 32, 16, 1024),
                 smem_desc_sw128(ks + (kk >> 2) * (kTcKTileBytes / 2) + (kk & 3) * 32, 16, 1024),
                 kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s);
        mma_commit(bar_ke + 8 * st);
        return true;
      };
      // Precise form, S(t) in two steps: Qhi.Khi + Qlo.Khi, then release the
      // Khi buffer; Qhi.Klo, then S is complete and the Klo buffer free.
      auto qk_hi = [&](int t) -> bool {
        if (!mbar_wait(bar_kf, t & 1, &abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t qs = sQ + part * kTcQBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tbase, smem_desc_sw128(qs + (kk >> 2) * (kTcQBytes / 2) + (kk & 3) * 32, 16, 1024),
                   smem_desc_sw128(sK + (kk >> 2) * (kTcKTileBytes / 2) + (kk & 3) * 32, 16, 1024),
                   kIdescQK, (part > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_ke);
        return true;
      };
      auto qk_lo = [&](int t) -> bool {
        if (!mbar_wait(bar_kf + 8, t & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t kl = sK + kTcKTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tbase, smem_desc_sw128(sQ + (kk >> 2) * (kTcQBytes / 2) + (kk & 3) * 32, 16, 1024),
                 smem_desc_sw128(kl + (kk >> 2) * (kTcKTileBytes / 2) + (kk & 3) * 32, 16, 1024),
                 kIdescQK, 1u);
        mma_commit(bar_s);
        mma_commit(bar_ke + 8);
        return true;
      };
      // O += P(t) V(t) over V stages [h0, h1) of the tile (halves of 8
      // k-steps, or quarters of 4); P(t) must be in TMEM
      auto pv_parts = [&](int t, int h0, int h1) -> bool {
        constexpr int kSteps = Plan::kVRows / 16;
        for (int h = h0; h < h1; ++h) {
          const int u = Plan::kVParts * t + h, vs = u % kTcVStages;
          if (!mbar_wait(bar_vf + 8 * vs, (u / kTcVStages) & 1, &abort_flag)) return false;
          tc_fence_after();
          const uint32_t v0 = sV + vs * Plan::kVBytes;
#pragma unroll
          for (int kk = 0; kk < kSteps; ++kk) {
            mma_ts(tbase + kColO, tbase + kColP + (Plan::kVRows / 2) * h + 8 * kk,
                   smem_desc_sw128(v0 + kk * 2048, Plan::kVBytes / 2, 1024), kIdescPV,
                   (t == 0 && h == 0 && kk == 0) ? 0u : 1u);
          }
          mma_commit(bar_ve + 8 * vs);
        }
        return true;
      };
      auto pv = [&](int t) -> bool {
        if (!mbar_wait(bar_p, t & 1, &abort_flag) || !pv_parts(t, 0, Plan::kVParts)) return false;
        mma_commit(bar_pfree);
        return true;
      };
      // Issue order: S(0); then for each t: S(t+1) (once the softmax has
      // loaded S(t)) and P.V(t) (once P(t) is in TMEM).
      if (kPrecise) {
        // S(t+1) is split around the first half of P.V(t), so that the V
        // quarters the second half needs can land while Qhi.Klo(t+1) runs
        ok = ok && qk_hi(0) && qk_lo(0);
        for (int t = 0; ok && t < ntiles; ++t) {
          const bool next = t + 1 < ntiles;
          ok = (!next || (mbar_wait(bar_sfree, t & 1, &abort_flag) && qk_hi(t + 1))) &&
               mbar_wait(bar_p, t & 1, &abort_flag) && pv_parts(t, 0, Plan::kVParts / 2) &&
               (!next || qk_lo(t + 1)) && pv_parts(t, Plan::kVParts / 2, Plan::kVParts);
          if (ok) mma_commit(bar_pfree);
        }
      } else {
        ok = ok && qk(0);
        for (int t = 0; ok && t < ntiles; ++t) {
          if (t + 1 < ntiles) {
            ok = mbar_wait(bar_sfree, t & 1, &abort_flag) && qk(t + 1);
            if (!ok) break;
          }
          ok = pv(t);
        }
      }
      if (!ok) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
      }
      // every MMA issued must retire before TMEM is released
      mma_commit(bar_done);
      (void)mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------- softmax warps ----
    const int hh = warp >> 2;                    // half: keys 128 hh .. 128 hh + 127 of each tile
    const int r = (warp & 3) * 32 + lane;        // row = TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tL = tbase + lane_bits;       // this lane's column 0
    const int32_t tloc = kTcPosPerCta * qb + (r >> 4);  // index in block
    const int32_t qp = ti.qa + (r >> 4);                // this row's position
    const int h = kGroup * g + (r & 15);
    const bool row_valid = tloc < p.n;  // rows past the block are padding
    const float sl2 = p.scale_log2;
    const int32_t wlo = local ? qp - p.window + 1 : INT32_MIN;  // lowest key in the window
    float mrow = -INFINITY, lhalf = 0.f;  // running max (same in both halves), this half's sum
    bool ok = true;

    // Every warp runs every tile's named barriers; after a timeout a warp
    // keeps doing so without touching TMEM (its results are dropped).
    for (int t = 0; t < ntiles; ++t) {
      // tcgen05.ld/st below are warp-collective: the whole warp goes on or stops
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_s, t & 1, &abort_flag));
      tc_fence_after();
      const int32_t kp0 = tile_kp0(ti, t) + 128 * hh;  // first key of this half
      const bool cache_tile = t < ti.ncache;
      const bool need_mask = (kp0 < 0) || (kp0 + 127 > ti.qa) ||
                             (local && kp0 < ti.qz - p.window + 1) ||
                             (cache_tile && kp0 + 127 >= ti.c0);
      uint32_t v[4][32];
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tL + 128 * hh + 32 * c, v[c]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) v[c][j] = 0xff800000u;
      }
      // S is in registers: the next tile's S = Q K^T may overwrite it
      tc_fence_before();
      mbar_arrive(bar_sfree);
      if (need_mask) {
        // keys kp0 + j are visible for j in [jlo, jhi]; the rest become -inf
        const int32_t jlo = max(max(wlo, 0), kp0) - kp0;
        const int32_t jhi = (cache_tile ? min(qp, ti.c0 - 1) : qp) - kp0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int32_t jj = 32 * c + j;
            v[c][j] = (jj < jlo || jj > jhi) ? 0xff800000u : v[c][j];
          }
      }
      float mx4[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float a = fmax3(__uint_as_float(v[c][0]), __uint_as_float(v[c][1]),
                        __uint_as_float(v[c][2]));
#pragma unroll
        for (int j = 3; j < 31; j += 2)
          a = fmax3(a, __uint_as_float(v[c][j]), __uint_as_float(v[c][j + 1]));
        mx4[c] = fmaxf(a, __uint_as_float(v[c][31]));
      }
      red_x[hh][r] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float mx = fmaxf(red_x[0][r], red_x[1][r]);
      asm volatile("bar.sync 2, 256;" ::: "memory");  // red_x is reused next tile
      const float mt = mx * sl2;  // scale > 0, so it commutes with max
      float alpha = 1.f;
      if (mt > mrow + kRescaleThreshold || (mrow == -INFINITY && mt != -INFINITY)) {
        if (mrow != -INFINITY) alpha = fast_exp2(mrow - mt);
        mrow = mt;
      }
      lhalf *= alpha;
      const float muse = (mrow == -INFINITY) ? 0.f : mrow;
      // P = 2^(s*scale*log2e - m) as bf16 pairs
      const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(-muse, -muse);
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint64_t x2 = fma_f32x2(f32x2(__uint_as_float(v[c][j]), __uint_as_float(v[c][j + 1])),
                                        sc2, nm2);
          float x0, x1;
          f32x2_split(x2, x0, x1);
          const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
          // the row sum adds the bf16 values P.V multiplies, so that the
          // normalisation matches them: with the running max held up to
          // 2^8 below the true one, the largest P is not 1 and its rounding
          // would otherwise scale a peaked row's output by up to 2^-9
          const uint32_t pr = pack_bf16x2(e0, e1);
          pk[c][j >> 1] = pr;
          ls2[(j >> 1) & 3] = add_f32x2(ls2[(j >> 1) & 3], f32x2(bf16lo(pr), bf16hi(pr)));
        }
      }
      {
        const uint64_t t2 = add_f32x2(add_f32x2(ls2[0], ls2[1]), add_f32x2(ls2[2], ls2[3]));
        float a0, a1;
        f32x2_split(t2, a0, a1);
        lhalf += a0 + a1;
      }
      // P(t) and the O rescale wait until P.V(t-1) has retired (it reads the
      // P columns and accumulates into O)
      if (t > 0)
        ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_pfree, (t - 1) & 1, &abort_flag));
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(tL + kColP + 64 * hh + 16 * c, pk[c]);
        // Rare: the running max grew by more than 2^8 -- rescale this half's
        // 64 columns of O.
        if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o32[32];
            tmem_ld32(tL + kColO + 64 * hh + 32 * c, o32);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o32[j] = __float_as_uint(__uint_as_float(o32[j]) * alpha);
            tmem_st32(tL + kColO + 64 * hh + 32 * c, o32);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p);
    }

    // ----------------------------------------------------------- epilogue ----
    if (ntiles > 0)
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_pfree, (ntiles - 1) & 1, &abort_flag));
    tc_fence_after();
    // the row sum: both halves' partial sums (same running max)
    red_x[hh][r] = lhalf;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float lrow = red_x[0][r] + red_x[1][r];
    ok = __all_sync(0xffffffffu, ok && !abort_flag);  // warp-uniform: it gates tcgen05.ld
    if (!ok && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
    const bool have = ok && ntiles > 0 && lrow > 0.f;
    const float inv = have ? 1.f / lrow : 0.f;
    const size_t orow = (static_cast<size_t>(b) * p.n + tloc) * kHq + h;
    uint32_t oa[2][32];  // this thread's 64 output dims, both loads in flight at once
    if (ok && ntiles > 0) {
      tmem_ld32(tL + kColO + 64 * hh, oa[0]);
      tmem_ld32(tL + kColO + 64 * hh + 32, oa[1]);
      tmem_wait_ld();
    }
    // Stage the normalised rows in shared memory (the key buffers: every
    // MMA has retired) -- a thread holds one row -- then store them with
    // coalesced 16-byte stores, a warp per row.  Rows are padded by 16
    // bytes so that the 32 rows a warp stages at once hit distinct banks.
    const bool part = p.splits > 1;
    constexpr int kStPadF = kD + 4;  // fp32 partial rows: 528 bytes
    constexpr int kStPadH = kD + 8;  // bf16 output rows: 272 bytes
    if (part) {
      float *st = reinterpret_cast<float *>(smem + Plan::kQ) + r * kStPadF + 64 * hh;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          reinterpret_cast<float4 *>(st + 32 * c)[q4] =
              make_float4(have ? __uint_as_float(oa[c][4 * q4 + 0]) * inv : 0.f,
                          have ? __uint_as_float(oa[c][4 * q4 + 1]) * inv : 0.f,
                          have ? __uint_as_float(oa[c][4 * q4 + 2]) * inv : 0.f,
                          have ? __uint_as_float(oa[c][4 * q4 + 3]) * inv : 0.f);
    } else {
      __nv_bfloat16 *st = reinterpret_cast<__nv_bfloat16 *>(smem + Plan::kQ) + r * kStPadH + 64 * hh;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t *a = oa[c];
          uint4 w;
          w.x = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 0]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 1]) * inv : 0.f);
          w.y = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 2]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 3]) * inv : 0.f);
          w.z = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 4]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 5]) * inv : 0.f);
          w.w = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 6]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 7]) * inv : 0.f);
          reinterpret_cast<uint4 *>(st + 32 * c)[q4] = w;
        }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    {
      const int tsm = threadIdx.x;  // 0..255 (the softmax warps)
      if (part) {
#pragma unroll 4
        for (int i = tsm; i < kTcRows * (kD / 4); i += 256) {
          const int rr = i >> 5, c4 = i & 31;
          const int32_t tl = kTcPosPerCta * qb + (rr >> 4);
          if (tl >= p.n) continue;
          const size_t orr = (static_cast<size_t>(b) * p.n + tl) * kHq + kGroup * g + (rr & 15);
          reinterpret_cast<float4 *>(p.part_o + (orr * p.splits + split) * kD)[c4] =
              reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(smem + Plan::kQ) +
                                               rr * kStPadF)[c4];
        }
      } else {
#pragma unroll 4
        for (int i = tsm; i < kTcRows * (kD / 8); i += 256) {
          const int rr = i >> 4, c8 = i & 15;
          const int32_t tl = kTcPosPerCta * qb + (rr >> 4);
          if (tl >= p.n) continue;
          const size_t orr = (static_cast<size_t>(b) * p.n + tl) * kHq + kGroup * g + (rr & 15);
          reinterpret_cast<uint4 *>(p.o + orr * kD)[c8] = reinterpret_cast<const uint4 *>(
              reinterpret_cast<const __nv_bfloat16 *>(smem + Plan::kQ) + rr * kStPadH)[c8];
        }
      }
    }
    if (p.splits > 1 && row_valid && hh == 0)
      p.part_lse[orow * p.splits + split] = have ? mrow + __log2f(lrow) : -INFINITY;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t launch_attn_tc(const TcParams &p, const CUtensorMap &tq, const CUtensorMap &tka,
                           const CUtensorMap &tva, const CUtensorMap &tkb, const CUtensorMap &tvb,
                           const CUtensorMap &tql, const CUtensorMap &tkl, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(p.qblocks * p.splits), kHkv, static_cast<unsigned>(p.batch));
  if (p.staged) {
    cudaError_t e =
        ensure_smem_attr(reinterpret_cast<const void *>(attn_tc_kernel<true>), kTcSmem, 5);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_tc_kernel<true>, grid, dim3(kTcThreads), kTcSmem, s, p, tq, tka, tva,
                      tkb, tvb, tql, tkl);
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(attn_tc_kernel<false>), kTcSmem, 1);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_tc_kernel<false>, grid, dim3(kTcThreads), kTcSmem, s, p, tq, tka, tva, tkb,
                    tvb, tql, tkl);
}

}  // namespace mg
