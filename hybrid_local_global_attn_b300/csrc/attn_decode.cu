// attn_decode.cu -- split-KV flash-decode of one query token per sequence in
// a global (full-context, no RoPE) layer.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// section 01; "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer",
// section "长上下文仍然带来计算开销"): for the query at position p, softmax
// attention over the keys at positions [0, p] of the linear cache, without
// RoPE; 16 query heads share one KV head.
//
// Design (HBM-bound: every K/V byte is read once):
//  * One CTA per (split, KV head, sequence), two CTAs per SM; split s of S
//    takes the 64-key tiles s, s + S, s + 2S, ... of [0, p], so that at any
//    moment the CTAs stream neighbouring tiles (contiguous runs per split
//    were ~2.5 % slower).
//  * A producer warp streams the tiles with TMA (128-byte swizzle, two
//    64-dim boxes per tile) through a 3-stage mbarrier ring; before the
//    dependency wait it warms L2 with the first tiles of the range the split
//    gets when the query sits at max_len - 1.
//  * Four consumer warps take 16 keys each of every tile.  The 16 query heads
//    of the KV group form the M = 16 side of mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate) for both Q.K^T and P.V; K and V fragments come from
//    ldmatrix / ldmatrix.trans of the swizzled tiles.  Online softmax in
//    base 2 with quad shuffles; row sums stay per thread until the end.
//  * The four warps merge in shared memory into the CTA's partial (o / l,
//    lse), written to the workspace; a combine kernel merges the splits.
//    With a single split per (sequence, KV head) -- large batches -- the
//    CTA writes the output itself and no combine runs.
//  * Optionally the token's own K/V is appended by the CTA whose split holds
//    its slot, before that tile is loaded (mg_append_decode).
//  * The cache is linear or paged (a page table maps each 256-multiple run
//    of positions of a sequence to a page of a shared pool); a 64-key tile
//    always lies inside one page.
#include "mg_internal.h"
#include "mg_ptx.cuh"
#include "mma_frag.cuh"

namespace mg {

namespace {

constexpr int kStages = kDecStages;
constexpr int kPageAhead = 128;  // paged cache: tiles whose pages are looked up together
// stages, barriers, the query tile [16 rows][256 B], + alignment slack
constexpr int kOffQ = kStages * kDecStageBytes + 256;
constexpr int kSmem = kOffQ + kGroup * kD * 2 + 1024;
static_assert(2 * 8 * kStages <= 256, "barriers fit before the query tile");

}  // namespace

__global__ void __launch_bounds__(kDecThreads, 2)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  constexpr int NS = kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ int32_t page_outer[kPageAhead];  // outer index of the CTA's first tiles (paged)
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NS * kDecStageBytes);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * NS;

  // MG_OVERLAP_NEXT with a single split (this kernel writes o itself, no
  // combine follows): the next kernel may begin at once
  const bool release_now = p.overlap != 0 && p.splits == 1;
  if (release_now) pdl_launch_dependents();
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
  if (warp == kDecWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    // Warm L2 with the CTA's first tiles while the previous kernel is still
    // running, one lane per tile (a paged cache's table loads then run side
    // by side); only a prefetch -- the loads that feed the math come after
    // pdl_wait().  (A paged cache's table may still be changing: a stale
    // entry only warms the wrong page.)
    static_assert(kDecPrefetchTiles <= 32, "one lane per prefetched tile");
    const int32_t pos = (split + lane * p.splits) * kDecTile;
    if (lane < kDecPrefetchTiles && pos < min(p.max_len, p.slots)) {
      int32_t r = pos, o = b * kHkv + g;
      if (p.map.table != nullptr) cache_coord(p.map, b, g, pos, &r, &o, nullptr);
      for (int x = 0; x < 2; ++x) {
        tma_prefetch_l2_3d(&tk, 64 * x, r, o);
        tma_prefetch_l2_3d(&tv, 64 * x, r, o);
      }
    }
  }
  __syncthreads();
  // Early start (caller's promise that no kernel still running writes the
  // cache or the positions): the position is read and the first stages are
  // issued before the dependency wait; everything an earlier kernel may
  // produce (q, the new row) and every write come after it.
  const bool early = p.early != 0;
  if (!early) {
    pdl_wait();
    if (!release_now) pdl_launch_dependents();
  }

  const int32_t pq = p.pos[b];
  const bool bad = pq < 0 || pq >= p.max_len || pq >= p.slots;
  const int32_t n_slots = bad ? 0 : pq + 1;
  const int32_t n_tiles_all = (n_slots + kDecTile - 1) / kDecTile;  // tiles of [0, p]
  const int ntiles = split < n_tiles_all ? (n_tiles_all - split + p.splits - 1) / p.splits : 0;
  const bool empty = ntiles == 0;
  // first slot of the CTA's t-th tile (keys at or past n_slots are masked)
  auto tile_pos = [&](int t) -> int32_t { return (split + t * p.splits) * kDecTile; };
  const size_t row0 = static_cast<size_t>(b) * kHq + g * kGroup;  // first query row of the group
  const bool fused_here = p.k_new != nullptr && !empty && (pq / kDecTile) % p.splits == split;
  // tiles issued before the wait (early start, linear cache): the first
  // stages, short of the tile that will hold the new row
  int npre = 0;
  if (early && warp == kDecWarps && lane == 0 && !empty && p.map.table == nullptr) {
    npre = min(NS, ntiles);
    if (fused_here) npre = min(npre, (pq / kDecTile) / p.splits);
    for (int t = 0; t < npre; ++t) {
      if (t == p.stall_tile) {
        npre = t;
        break;
      }
      const uint32_t dst = smem_base + t * kDecStageBytes;
      const uint32_t fb = bar_full + 8 * t;
      const int32_t row = tile_pos(t);
      mbar_arrive_expect_tx(fb, kDecStageBytes);
      tma_load_3d(dst, &tk, fb, 0, row, b * kHkv + g);
      tma_load_3d(dst + 8192, &tk, fb, 64, row, b * kHkv + g);
      tma_load_3d(dst + 16384, &tv, fb, 0, row, b * kHkv + g);
      tma_load_3d(dst + 24576, &tv, fb, 64, row, b * kHkv + g);
    }
  }
  if (early) {
    pdl_wait();
    if (!release_now) pdl_launch_dependents();
  }
  if (bad && split == 0 && threadIdx.x == 0) set_err(p.err, MG_DERR_POSITION);
  // this CTA's partial of row r: o already divided by its softmax sum, and lse
  auto part_o = [&](int r, int d) -> float & {
    return p.part_o[((row0 + r) * p.splits + split) * kD + d];
  };
  auto part_lse = [&](int r) -> float & { return p.part_lse[(row0 + r) * p.splits + split]; };

  bool ok = true;
  if (warp == kDecWarps) {
    // ------------------------------------------------ TMA producer warp ----
    if (!empty) {
      // Fused append: the query token's K/V row lands in its slot before the
      // tile that holds the slot is read (the TMA read goes through the async
      // proxy, hence the proxy fence after the stores).
      if (fused_here) {
        const size_t src = (static_cast<size_t>(b) * kHkv + g) * kD;
        int32_t r, o;
        cache_coord(p.map, b, g, pq, &r, &o, lane == 0 ? p.err : nullptr);
        const size_t dst = (static_cast<size_t>(o) * p.map.rows + r) * kD;
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
      // A tile never straddles two pages (64 | 256 | page size).  Paged
      // cache: the warp's lanes look up the pages of the CTA's first
      // kPageAhead tiles together (one round of parallel table loads); a
      // later tile's page is fetched one tile ahead by the issuing lane.
      const bool paged = p.map.table != nullptr;
      if (paged) {
        for (int t = lane; t < min(ntiles, kPageAhead); t += 32) {
          int32_t r, o;
          cache_coord(p.map, b, g, tile_pos(t), &r, &o, p.err);
          page_outer[t] = o;
        }
        __syncwarp();
      }
      if (lane == 0) {
        int issued = npre;
        int32_t nrow = 0, nouter = 0;
        if (paged && kPageAhead < ntiles) cache_coord(p.map, b, g, tile_pos(kPageAhead), &nrow, &nouter, p.err);
        for (int t = npre; t < ntiles; ++t) {
          const int st = t % NS;
          if (t == p.stall_tile) break;  // self-test: tiles from here on never arrive
          int32_t row = tile_pos(t), outer = b * kHkv + g;
          if (paged && t < kPageAhead) {
            row %= p.map.rows;
            outer = page_outer[t];
          } else if (paged) {
            row = nrow;
            outer = nouter;
            if (t + 1 < ntiles) cache_coord(p.map, b, g, tile_pos(t + 1), &nrow, &nouter, p.err);
          }
          if (t >= NS &&
              !mbar_wait(bar_empty + 8 * st, ((t / NS) - 1) & 1, &abort_flag, p.wait_ns)) {
            abort_flag = 1;
            set_err(p.err, MG_DERR_TIMEOUT);
            break;
          }
          const uint32_t dst = smem_base + st * kDecStageBytes;
          const uint32_t fb = bar_full + 8 * st;
          mbar_arrive_expect_tx(fb, kDecStageBytes);
          tma_load_3d(dst, &tk, fb, 0, row, outer);
          tma_load_3d(dst + 8192, &tk, fb, 64, row, outer);
          tma_load_3d(dst + 16384, &tv, fb, 0, row, outer);
          tma_load_3d(dst + 24576, &tv, fb, 64, row, outer);
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

    // Q fragments (A operand, 16 heads x 128 dims): the group's 4 KB of
    // query rows with coalesced 16-byte loads into shared memory (rows 256
    // bytes apart, 16-byte chunks XOR-swizzled by the row), then ldmatrix
    uint32_t qf[8][4];
    {
      const uint32_t qs = smem_base + kOffQ;
      const int qr = tid >> 3;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = (tid & 7) + 8 * h;
        const uint4 v4 = __ldg(reinterpret_cast<const uint4 *>(p.q + (row0 + qr) * kD) + c);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qs + qr * 256 + ((c ^ (qr & 7)) << 4)),
                     "r"(v4.x), "r"(v4.y), "r"(v4.z), "r"(v4.w)
                     : "memory");
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
      const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int chunk = 2 * ks + (lane >> 4);
        ldsm_x4(qs + row * 256 + ((chunk ^ (row & 7)) << 4), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
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
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar_full + 8 * st, (t / NS) & 1, &abort_flag, p.wait_ns))) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
        ok = false;
        break;
      }
      const int32_t key0 = tile_pos(t) + warp * 16;  // slot of this warp's first key
      if (key0 < n_slots) {
        const uint32_t kbase = smem_base + st * kDecStageBytes;
        const uint32_t vbase = kbase + 16384;
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
            sacc[j][e] = (key < n_slots) ? sacc[j][e] * sl2 : -INFINITY;
          }
        }
        float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
        float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: key0 < n_slots
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
    // sum the four scaled slices into this split's partial
#pragma unroll 4
    for (int i = tid; i < kGroup * kD; i += kDecWarps * 32) {
      const int r = i / kD, d = i % kD;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) acc += mo[(w * kGroup + r) * kRowPad + d];
      if (p.splits == 1)
        p.o[(row0 + r) * kD + d] = __float2bfloat16_rn(acc);  // the only split: final
      else
        part_o(r, d) = acc;
    }
    if (warp == 0 && tq == 0 && p.splits > 1) {
      part_lse(gr) = Lr[0] > 0.f ? Mr[0] + __log2f(Lr[0]) : -INFINITY;
      part_lse(gr + 8) = Lr[1] > 0.f ? Mr[1] + __log2f(Lr[1]) : -INFINITY;
    }
  } else {
    // no keys for this split: lse = -inf, o = 0
    for (int i = threadIdx.x; i < kGroup * kD; i += kDecWarps * 32) {
      if (p.splits == 1)
        p.o[(row0 + i / kD) * kD + i % kD] = __float2bfloat16_rn(0.f);
      else
        part_o(i / kD, i % kD) = 0.f;
    }
    if (threadIdx.x < kGroup && p.splits > 1) part_lse(threadIdx.x) = -INFINITY;
  }
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t s) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(decode_kernel), kSmem, 0);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, kHkv, p.batch);
  return launch_pdl(decode_kernel, grid, dim3(kDecThreads), kSmem, s, p, tk, tv);
}

}  // namespace mg
