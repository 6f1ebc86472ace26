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
// head).  Key tiles hold 128 keys and are aligned to c0, so a tile never
// straddles the cache and the block.
//
// Shared-memory bandwidth (128 B/cycle) is the tight resource of a
// single-CTA tcgen05 pipeline: per 128x128 tile the TMA fill (64 KB), the
// K operand (32 KB) and the V operand (32 KB) already take ~1000 cycles.  So
// the query tile lives in TMEM and is the A operand of S = Q K^T, as P is of
// O += P V; only K and V are read from shared memory.
//
// Warp roles (320 threads):
//   warps 0-3  softmax of keys 0..63 of every key tile (thread = row = lane)
//   warps 4-7  softmax of keys 64..127 of the same rows; the two halves
//              exchange their row maxima once per tile
//   warp 8     TMA producer (Q once; K in a 2-deep ring, V in a 4-deep ring:
//              V of a tile is consumed a softmax after its K)
//   warp 9     TMEM owner and single-thread MMA issuer
// TMEM (512 columns): S_0, S_1 (double-buffered scores, fp32 128 cols each;
// P overwrites the first 64 columns as packed bf16), O (fp32 128 cols), Q
// (bf16 pairs, 64 cols).  S = Q K^T of tile t + 1 runs while the softmax
// works on tile t.
// Per key tile: S = Q K^T (M128 N128 K16 x 8, A from TMEM), softmax in
// registers with a lazily rescaled running max (rescale only when the max
// grows by more than 2^8), P back to TMEM, O += P V (A from TMEM, V as an
// MN-major operand).
// Splits (verify): the cache part is cut across CTAs; each writes (o/l, lse)
// and the combine kernel merges them.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct TileInfo {
  int32_t c0, qa, qz;     // block start, first and last valid query position
  int32_t ncache, nnew;   // tiles from the cache part / the block part
  int32_t u_begin, v_lo;  // first cache tile index (from c0 down), first block tile
};

__device__ __forceinline__ int32_t tile_kp0(const TileInfo &ti, int t) {
  if (t < ti.ncache) return ti.c0 - kTcKeys * (ti.u_begin + t + 1);
  return ti.c0 + kTcKeys * (ti.v_lo + (t - ti.ncache));
}

}  // namespace

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tka, const __grid_constant__ CUtensorMap tva,
                   const __grid_constant__ CUtensorMap tkb,
                   const __grid_constant__ CUtensorMap tvb) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_base_slot;
  __shared__ float red_x[2][kTcRows];  // per tile: the two halves' row maxima
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase;                        // 32 KB (copied into TMEM)
  const uint32_t sK = sbase + kTcQBytes;            // K ring: stage s at +32K*s
  const uint32_t sV = sK + kTcKStages * kTcTileBytes;  // V ring
  const uint32_t sBar = sV + kTcVStages * kTcTileBytes;
  // barrier addresses
  const uint32_t bar_q = sBar;                             // Q in shared memory
  const uint32_t bar_kf = sBar + 8;                        // [kTcKStages] K full
  const uint32_t bar_ke = bar_kf + 8 * kTcKStages;         // [kTcKStages] K stage free
  const uint32_t bar_vf = bar_ke + 8 * kTcKStages;         // [kTcVStages] V full
  const uint32_t bar_ve = bar_vf + 8 * kTcVStages;         // [kTcVStages] V stage free
  const uint32_t bar_s = bar_ve + 8 * kTcVStages;          // [2] S buffer ready
  const uint32_t bar_p = bar_s + 16;                       // [2] P ready (256 arrivals)
  const uint32_t bar_qt = bar_p + 16;                      // Q in TMEM (256 arrivals)
  const uint32_t bar_o = bar_qt + 8;                       // O final
  const uint32_t bar_done = bar_o + 8;                     // all MMAs retired

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
  ti.qa = ti.c0 + kTcPosPerCta * qb;
  ti.qz = min(ti.qa + kTcPosPerCta - 1, ti.c0 + p.n - 1);
  ti.ncache = ti.nnew = ti.u_begin = ti.v_lo = 0;
  if (!bad) {
    const int32_t lo = local ? max(0, ti.qa - p.window + 1) : 0;
    const int32_t U = ti.c0 > lo ? (ti.c0 - lo + kTcKeys - 1) / kTcKeys : 0;
    ti.u_begin = static_cast<int32_t>(static_cast<int64_t>(split) * U / p.splits);
    const int32_t u_end = static_cast<int32_t>(static_cast<int64_t>(split + 1) * U / p.splits);
    ti.ncache = u_end - ti.u_begin;
    if (split == p.splits - 1) {
      ti.v_lo = local ? max(0, ti.qa - p.window + 1 - ti.c0) / kTcKeys : 0;
      const int32_t v_hi = (ti.qz - ti.c0) / kTcKeys;
      ti.nnew = v_hi - ti.v_lo + 1;
    }
  }
  const int ntiles = ti.ncache + ti.nnew;

  if (threadIdx.x == 0) {
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s + 8 * i, 1);
      mbar_init(bar_p + 8 * i, 256);
    }
    mbar_init(bar_qt, 256);
    mbar_init(bar_o, 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&tmem_base_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_slot;
  constexpr uint32_t kColO = 256, kColQ = 384;

  if (warp == 8) {
    // ------------------------------------------------------- producer ----
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tka);
      tma_prefetch_desc(&tva);
      tma_prefetch_desc(&tkb);
      tma_prefetch_desc(&tvb);
      const int32_t q_t0 = kTcPosPerCta * qb;  // position index within the block
      mbar_arrive_expect_tx(bar_q, kTcQBytes);
      for (int x = 0; x < 2; ++x)
        tma_load_4d(sQ + x * (kTcQBytes / 2), &tq, bar_q, 64 * x, kGroup * g, q_t0, b);
      int issued_k = 0, issued_v = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int32_t kp0 = tile_kp0(ti, t);
        const bool from_cache = t < ti.ncache;
        // one 128-key tile of K or V into dst, completing on fb
        auto load_tile = [&](bool is_v, uint32_t dst, uint32_t fb) {
          const CUtensorMap *ma = is_v ? &tva : &tka;
          const CUtensorMap *mb = is_v ? &tvb : &tkb;
          mbar_arrive_expect_tx(fb, kTcTileBytes);
          for (int x = 0; x < 2; ++x) {
            const uint32_t d = dst + x * (kTcTileBytes / 2);
            if (p.staged)
              tma_load_3d(d, ma, fb, 64 * x, kp0 - ti.c0 + kWindow, b * kHkv + g);
            else if (from_cache)
              tma_load_3d(d, ma, fb, 64 * x, kp0, b * kHkv + g);
            else
              tma_load_4d(d, mb, fb, 64 * x, g, kp0 - ti.c0, b);
          }
        };
        // K of tile t reuses the stage of tile t - kTcKStages once its
        // S = Q K^T has run; V reuses the stage of tile t - kTcVStages once
        // its P.V has run
        const int ks = t % kTcKStages, vs = t % kTcVStages;
        if (t >= kTcKStages &&
            !mbar_wait(bar_ke + 8 * ks, ((t / kTcKStages) - 1) & 1, &abort_flag)) {
          abort_flag = 1;
          set_err(p.err, MG_DERR_TIMEOUT);
          break;
        }
        load_tile(false, sK + ks * kTcTileBytes, bar_kf + 8 * ks);
        ++issued_k;
        if (t >= kTcVStages &&
            !mbar_wait(bar_ve + 8 * vs, ((t / kTcVStages) - 1) & 1, &abort_flag)) {
          abort_flag = 1;
          set_err(p.err, MG_DERR_TIMEOUT);
          break;
        }
        load_tile(true, sV + vs * kTcTileBytes, bar_vf + 8 * vs);
        ++issued_v;
      }
      // no copies may be in flight when the CTA retires
      (void)mbar_wait(bar_q, 0, nullptr);
      for (int t = max(0, issued_k - kTcKStages); t < issued_k; ++t)
        (void)mbar_wait(bar_kf + 8 * (t % kTcKStages), (t / kTcKStages) & 1, nullptr);
      for (int t = max(0, issued_v - kTcVStages); t < issued_v; ++t)
        (void)mbar_wait(bar_vf + 8 * (t % kTcVStages), (t / kTcVStages) & 1, nullptr);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(bar_qt, 0, &abort_flag);  // Q copied into TMEM by the softmax warps
      // S_{t&1} = Q K(t)^T, Q from TMEM
      auto qk = [&](int t) -> bool {
        const int st = t % kTcKStages;
        if (!mbar_wait(bar_kf + 8 * st, (t / kTcKStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t ks = sK + st * kTcTileBytes;
        const uint32_t tS = tbase + 128 * (t & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTcTileBytes / 2) + (kk & 3) * 32;
          mma_ts(tS, tbase + kColQ + 8 * kk, smem_desc_sw128(ks + off, 16, 1024), kIdescQK,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s + 8 * (t & 1));
        mma_commit(bar_ke + 8 * st);
        return true;
      };
      // O += P(t) V(t), P from the first half of S_{t&1}
      auto pv = [&](int t) -> bool {
        const int st = t % kTcVStages, e = t & 1;
        if (!mbar_wait(bar_p + 8 * e, (t >> 1) & 1, &abort_flag)) return false;
        if (!mbar_wait(bar_vf + 8 * st, (t / kTcVStages) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t vs = sV + st * kTcTileBytes;
        const uint32_t tS = tbase + 128 * e;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_ts(tbase + kColO, tS + 8 * kk, smem_desc_sw128(vs + kk * 2048, kTcTileBytes / 2, 1024),
                 kIdescPV, (t == 0 && kk == 0) ? 0u : 1u);
        }
        mma_commit(bar_ve + 8 * st);
        if (t == ntiles - 1) mma_commit(bar_o);
        return true;
      };
      // Issue order: S(0), S(1), then P.V(t) and S(t+2) for t = 0, 1, ...
      // S(t+2) reuses the TMEM of S(t) = P(t), so it goes after P.V(t); the
      // MMAs of one thread run in issue order.
      ok = ok && qk(0);
      if (ntiles > 1) ok = ok && qk(1);
      for (int t = 0; ok && t < ntiles; ++t) {
        ok = pv(t);
        if (ok && t + 2 < ntiles) ok = qk(t + 2);
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
    const int hh = warp >> 2;                    // half: keys 64 hh .. 64 hh + 63 of each tile
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

    // Q row r, dims 64 hh .. 64 hh + 63 (swizzled box hh of the Q tile),
    // into TMEM columns kColQ + 32 hh .. as bf16 pairs
    if (ntiles > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, &abort_flag));
      uint32_t qv[32];
      const uint32_t box = sQ + hh * (kTcQBytes / 2) + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t a0, a1, a2, a3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                     : "r"(box + ((c ^ (r & 7)) << 4)));
        qv[4 * c] = a0;
        qv[4 * c + 1] = a1;
        qv[4 * c + 2] = a2;
        qv[4 * c + 3] = a3;
      }
      tmem_st32(tL + kColQ + 32 * hh, qv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_qt);
    }

    // Every warp runs every tile's two named barriers; after a timeout a warp
    // keeps doing so without touching TMEM (its results are dropped).
    for (int t = 0; t < ntiles; ++t) {
      const int e = t & 1;
      const uint32_t tS = tL + 128 * e;
      // tcgen05.ld/st below are warp-collective: the whole warp goes on or stops
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_s + 8 * e, (t >> 1) & 1, &abort_flag));
      tc_fence_after();
      const int32_t kp0 = tile_kp0(ti, t) + 64 * hh;  // first key of this half
      const bool need_mask = (kp0 < 0) || (kp0 + 63 > ti.qa) ||
                             (local && kp0 < ti.qz - p.window + 1);
      uint32_t v[2][32];
      if (ok) {
        tmem_ld32(tS + 64 * hh, v[0]);
        tmem_ld32(tS + 64 * hh + 32, v[1]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[0][j] = v[1][j] = 0xff800000u;
      }
      if (need_mask) {
        // keys kp0 + j are visible for j in [jlo, jhi]; the rest become -inf
        const int32_t jlo = max(max(wlo, 0), kp0) - kp0;
        const int32_t jhi = qp - kp0;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int32_t jj = 32 * c + j;
            v[c][j] = (jj < jlo || jj > jhi) ? 0xff800000u : v[c][j];
          }
      }
      float mx2[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float a = fmax3(__uint_as_float(v[c][0]), __uint_as_float(v[c][1]),
                        __uint_as_float(v[c][2]));
#pragma unroll
        for (int j = 3; j < 31; j += 2)
          a = fmax3(a, __uint_as_float(v[c][j]), __uint_as_float(v[c][j + 1]));
        mx2[c] = fmaxf(a, __uint_as_float(v[c][31]));
      }
      // the row's max over both halves (every S value is in registers, so P
      // may overwrite S after this barrier)
      red_x[hh][r] = fmaxf(mx2[0], mx2[1]);
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
      // P = 2^(s*scale*log2e - m) as bf16 pairs: keys 64 hh + 2c.. -> column 32 hh + c
      const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(-muse, -muse);
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint64_t x2 = fma_f32x2(f32x2(__uint_as_float(v[c][j]), __uint_as_float(v[c][j + 1])),
                                        sc2, nm2);
          float x0, x1;
          f32x2_split(x2, x0, x1);
          const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
          ls2[(j >> 1) & 3] = add_f32x2(ls2[(j >> 1) & 3], f32x2(e0, e1));
          pk[j >> 1] = pack_bf16x2(e0, e1);
        }
        if (ok) tmem_st16(tS + 32 * hh + 16 * c, pk);
      }
      {
        const uint64_t t2 = add_f32x2(add_f32x2(ls2[0], ls2[1]), add_f32x2(ls2[2], ls2[3]));
        float a0, a1;
        f32x2_split(t2, a0, a1);
        lhalf += a0 + a1;
      }
      // Rare: the running max grew by more than 2^8 -- rescale O in TMEM
      // (this half's 64 columns).  S(t) was issued after P.V(t-2), so that
      // one has retired, but P.V(t-1) may still run: wait for its V stage
      // release first.  The next P.V waits for this tile's P arrival below.
      if (ok && t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const int pst = (t - 1) % kTcVStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar_ve + 8 * pst, ((t - 1) / kTcVStages) & 1, &abort_flag)) && ok;
        tc_fence_after();
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
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p + 8 * e);
    }

    // ----------------------------------------------------------- epilogue ----
    if (ok && ntiles > 0 && !__all_sync(0xffffffffu, mbar_wait(bar_o, 0, &abort_flag))) ok = false;
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
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int d0 = 64 * hh + 32 * c;  // first dim of this 32-column chunk
      uint32_t a[32];
      if (ok && ntiles > 0) {
        tmem_ld32(tL + kColO + d0, a);
        tmem_wait_ld();
      }
      if (!row_valid) continue;
      if (p.splits == 1) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow * kD + d0);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 0]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 1]) * inv : 0.f);
          w.y = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 2]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 3]) * inv : 0.f);
          w.z = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 4]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 5]) * inv : 0.f);
          w.w = pack_bf16x2(have ? __uint_as_float(a[8 * q4 + 6]) * inv : 0.f,
                            have ? __uint_as_float(a[8 * q4 + 7]) * inv : 0.f);
          dst[q4] = w;
        }
      } else {
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + (orow * p.splits + split) * kD + d0);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst[q4] = make_float4(have ? __uint_as_float(a[4 * q4 + 0]) * inv : 0.f,
                                have ? __uint_as_float(a[4 * q4 + 1]) * inv : 0.f,
                                have ? __uint_as_float(a[4 * q4 + 2]) * inv : 0.f,
                                have ? __uint_as_float(a[4 * q4 + 3]) * inv : 0.f);
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
                           cudaStream_t s) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(attn_tc_kernel), kTcSmem, 1);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.qblocks * p.splits), kHkv, static_cast<unsigned>(p.batch));
  return launch_pdl(attn_tc_kernel, grid, dim3(kTcThreads), kTcSmem, s, p, tq, tka, tva, tkb, tvb);
}

}  // namespace mg
