// attn_decode_e4m3.cu -- split-KV flash-decode of one query token per
// sequence in a global layer whose cache holds FP8 (OCP E4M3) codes.
//
// What it computes: the same attention as the bf16 decode kernel ("深度拆解
// Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？", section 01; "Tomas
// Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer", sections
// "长上下文仍然带来计算开销" and, for quantising the cache,
// "窄缓存为长上下文留出空间"), over keys and values that are the codes times a
// power-of-two scale per KV head.  Half the bytes per key (512 instead of
// 1024), so the HBM-bound pass takes about half the time.
//
// Layout (per sequence and KV head): K codes [pos][128]; V codes transposed
// per 64-position tile, [tile][dim][64], positions inside each 16-position
// group in the column order c(j) = 4 ((j % 8) / 2) + 2 (j / 8) + j % 2.
//
// Design (differences from the bf16 kernel):
//  * Split s of S takes the 128-key tiles s, s + S, s + 2S, ... (as the
//    bf16 kernel does with its 64-key tiles).
//  * A stage is 128 keys: 16 KB of K (one 128-byte-swizzled box) + 16 KB
//    of V (one 64-byte-swizzled box of two transposed tiles); 3 stages in
//    flight, 2 CTAs per SM.  Each of the 4 consumer warps takes 32 keys of a
//    stage as two independent 16-key groups (twice the bf16 kernel's keys
//    per warp: the conversions make the per-key work larger, and two groups
//    give each warp independent chains to interleave).
//  * e4m3 -> f16 is exact; the tensor-core products run in f16
//    (mma.sync m16n8k16, fp32 accumulate).  The query is moved to f16 with a
//    power-of-two factor per row that puts its largest element in [2^14,
//    2^15): exact for every element down to 2^-29 of the largest, and the
//    factor is folded into the row's score scale with the K scale.  P is
//    stored as f16 (more precise than bf16 for values in (0, 1]).
//  * Plain ldmatrix of the codes: a lane's 32-bit fragment holds 4
//    consecutive bytes.  For Q.K^T those are dims 4t..4t+3 of one key: the
//    reduction dims are used in the order (4t, 4t+1 | 4t+2, 4t+3) for
//    (k = 2t, 2t+1 | 2t+8, 2t+9), and the query fragments are loaded in the
//    same order.  For P.V they are 4 columns of one dim of the transposed
//    tile, which the column order above fills with keys 2t, 2t+1, 8+2t, 9+2t
//    -- exactly the keys whose probabilities the Q.K^T accumulators of a
//    lane hold, so P goes from accumulators to A fragments unchanged.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mg_internal.h"
#include "mg_ptx.cuh"
#include "mma_frag.cuh"

namespace mg {

namespace {

constexpr int NS = kE4m3Stages;
constexpr int kT = kE4m3Tile;                  // keys per stage (32 per consumer warp)
constexpr int kVT = 64;                        // positions per transposed V tile (layout)
constexpr int kKBytes = kT * kD;               // 16 KB of K codes per stage
constexpr int kStage = 2 * kKBytes;            // + 16 KB of V codes (two transposed tiles)
// stages, barriers, the query tile [16 rows][256 B], + alignment slack
constexpr int kOffQ = NS * kStage + 256;
constexpr int kSmem = kOffQ + kGroup * kD * 2 + 1024;
static_assert(2 * 8 * NS <= 256, "barriers fit before the query tile");

// Four e4m3 codes (bytes 0..3 of x) -> two f16 x2 (bytes 0, 1 and bytes 2,
// 3; lower byte to the lower half), exact: one conversion per 16-bit half,
// taken straight from the register's halves.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t x, uint32_t &lo, uint32_t &hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

constexpr float kLazyRescale = 8.0f;  // log2 units

// 2^e as a float (e in the normal range)
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// 1 / s for a power of two s = 2^e with -126 <= e <= 126: the exponent
// field flips around 127 (exact, unlike a reciprocal instruction).
__device__ __forceinline__ float pow2_recip(float s) {
  return __int_as_float(0x7F000000 - __float_as_int(s));
}

}  // namespace

__global__ void __launch_bounds__(kDecThreads, 2)
    decode_e4m3_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NS * kStage);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * NS;
  const int32_t vtiles = p.slots / kVT;  // transposed V tiles per (sequence, head)
  const int32_t c2 = b * kHkv + g;

  // MG_OVERLAP_NEXT with a single split (this kernel writes o itself, no
  // combine follows): the next kernel may begin at once
  const bool release_now = p.overlap != 0 && p.splits == 1;
  if (release_now) pdl_launch_dependents();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kDecWarps);
    }
    fence_mbar_init();
  }
  if (warp == kDecWarps && lane == 0) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    // warm L2 with the first tiles of the range the split gets when the
    // query sits at max_len - 1 (a prefetch only)
    const int32_t lim = min(p.max_len, p.slots);
    for (int t = 0; t < kE4m3PrefetchTiles; ++t) {
      const int32_t row = (split + t * p.splits) * kT;
      if (row >= lim) break;
      tma_prefetch_l2_3d(&tk, 0, row, c2);
      tma_prefetch_l2_4d(&tv, 0, 0, row / kVT, c2);
    }
  }
  __syncthreads();
  pdl_wait();
  if (!release_now) pdl_launch_dependents();

  const int32_t pq = p.pos[b];
  const bool bad = pq < 0 || pq >= p.max_len || pq >= p.slots;
  const int32_t n_slots = bad ? 0 : pq + 1;
  // split s of S takes the tiles s, s + S, s + 2S, ... of [0, p]: at any
  // moment the CTAs stream neighbouring tiles
  const int32_t n_tiles_all = (n_slots + kT - 1) / kT;
  const int ntiles = split < n_tiles_all ? (n_tiles_all - split + p.splits - 1) / p.splits : 0;
  const bool empty = ntiles == 0;
  auto tile_pos = [&](int t) -> int32_t { return (split + t * p.splits) * kT; };
  const size_t row0 = static_cast<size_t>(b) * kHq + g * kGroup;
  if (bad && split == 0 && threadIdx.x == 0) set_err(p.err, MG_DERR_POSITION);
  auto part_o = [&](int r, int d) -> float & {
    return p.part_o[((row0 + r) * p.splits + split) * kD + d];
  };
  auto part_lse = [&](int r) -> float & { return p.part_lse[(row0 + r) * p.splits + split]; };

  const bool fused_here = p.k_new != nullptr && !empty && (pq / kT) % p.splits == split;
  bool ok = true;
  if (warp == kDecWarps) {
    // ------------------------------------------------ TMA producer warp ----
    if (!empty) {
      if (fused_here) {
        // The token's own K/V, quantised, into its slot before the tile that
        // holds it is read.  Lane l < 16: dims 8l..8l+7 of K; lane l >= 16:
        // dims 8(l-16).. of V (one byte per dim row of the transposed tile).
        const int c = lane & 15;
        const bool is_v = lane >= 16;
        const __nv_bfloat16 *src = (is_v ? p.v_new : p.k_new) + (static_cast<size_t>(b) * kHkv + g) * kD + 8 * c;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src));
        const float mul = pow2_recip(is_v ? p.v_scale[g] : p.k_scale[g]);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t codes[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = bf16lo(w[i]) * mul, hi = bf16hi(w[i]) * mul;
          const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
          codes[i >> 1] |= (two & 0xFFFFu) << (16 * (i & 1));
        }
        if (!is_v) {
          uint8_t *dst = reinterpret_cast<uint8_t *>(p.k_cache) +
                         (static_cast<size_t>(c2) * p.slots + pq) * kD + 8 * c;
          *reinterpret_cast<uint2 *>(dst) = make_uint2(codes[0], codes[1]);
        } else {
          const int j = pq % 16;
          const int col = 16 * ((pq % kVT) / 16) + 4 * ((j % 8) / 2) + 2 * (j / 8) + j % 2;
          uint8_t *dst = reinterpret_cast<uint8_t *>(p.v_cache) +
                         (static_cast<size_t>(c2) * vtiles + pq / kVT) * (kD * kVT) +
                         static_cast<size_t>(8 * c) * kVT + col;
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i * kVT] = static_cast<uint8_t>(codes[i >> 2] >> (8 * (i & 3)));
        }
        fence_proxy_async_global();
        __syncwarp();
      }
      if (lane == 0) {
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
          const int st = t % NS;
          if (t >= NS && !mbar_wait(bar_empty + 8 * st, ((t / NS) - 1) & 1, &abort_flag)) {
            abort_flag = 1;
            set_err(p.err, MG_DERR_TIMEOUT);
            break;
          }
          const uint32_t dst = smem_base + st * kStage;
          const uint32_t fb = bar_full + 8 * st;
          const int32_t row = tile_pos(t);
          mbar_arrive_expect_tx(fb, kStage);
          tma_load_3d(dst, &tk, fb, 0, row, c2);                   // 128 keys x 128 dims
          tma_load_4d(dst + kKBytes, &tv, fb, 0, 0, row / kVT, c2);  // two transposed tiles
          ++issued;
        }
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

    // Q fragments in f16: chunk ks covers dims 16ks..16ks+15 taken in the
    // order (4tq, 4tq+1 | 4tq+2, 4tq+3); rows gr (head gr) and gr + 8.
    uint32_t qf[8][4];
    float sl2[2];
    {
      // the group's 4 KB of query rows with coalesced 16-byte loads into
      // shared memory (rows 256 bytes apart, 16-byte chunks XOR-swizzled by
      // the row), then each lane's 8-byte pieces from there
      const uint32_t qs = smem_base + kOffQ;
      {
        const int qrow = tid >> 3;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = (tid & 7) + 8 * h2;
          const uint4 v4 = __ldg(reinterpret_cast<const uint4 *>(p.q + (row0 + qrow) * kD) + c);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qs + qrow * 256 + ((c ^ (qrow & 7)) << 4)),
                       "r"(v4.x), "r"(v4.y), "r"(v4.z), "r"(v4.w)
                       : "memory");
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
      }
      uint2 raw[2][8];
      float amax[2] = {0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int row = gr + 8 * h, chunk = 2 * ks + (tq >> 1);
          asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                       : "=r"(raw[h][ks].x), "=r"(raw[h][ks].y)
                       : "r"(qs + row * 256 + ((chunk ^ (row & 7)) << 4) + 8 * (tq & 1)));
          amax[h] = fmaxf(amax[h], fmaxf(fmaxf(fabsf(bf16lo(raw[h][ks].x)), fabsf(bf16hi(raw[h][ks].x))),
                                         fmaxf(fabsf(bf16lo(raw[h][ks].y)), fabsf(bf16hi(raw[h][ks].y)))));
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        amax[h] = fmaxf(amax[h], __shfl_xor_sync(0xffffffffu, amax[h], 1));
        amax[h] = fmaxf(amax[h], __shfl_xor_sync(0xffffffffu, amax[h], 2));
        // 2^sh puts the row's largest element in [2^14, 2^15)
        const int e = amax[h] > 0.f ? ((__float_as_int(amax[h]) >> 23) & 0xFF) - 127 : 0;
        const int sh = min(max(14 - e, -126), 126);
        const float f = exp2i(sh);
        sl2[h] = p.scale_log2 * p.k_scale[g] * exp2i(-sh);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qf[ks][h] = pack_f16x2(bf16lo(raw[h][ks].x) * f, bf16hi(raw[h][ks].x) * f);
          qf[ks][h + 2] = pack_f16x2(bf16lo(raw[h][ks].y) * f, bf16hi(raw[h][ks].y) * f);
        }
      }
    }

    float oacc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // ldmatrix lane -> row addresses.  K: matrix j = lane / 8 covers keys
    // 8 (j & 1) + (lane & 7) of a 16-key group, chunk 2 kk + (j >> 1).  V:
    // matrix j covers dim rows 8 (4 q + j) + (lane & 7) of a transposed tile.
    const uint32_t k_row = (((lane >> 3) & 1) << 3) + (lane & 7);
    const uint32_t k_chi = lane >> 4;
    const uint32_t v_row = lane;

    for (int t = 0; t < ntiles; ++t) {
      const int st = t % NS;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (t / NS) & 1, &abort_flag))) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
        ok = false;
        break;
      }
      // this warp: keys key0 .. key0 + 31 of the tile, as two groups of 16
      const int32_t key0 = tile_pos(t) + warp * 32;
      if (key0 < n_slots) {
        const uint32_t kbase = smem_base + st * kStage;
        const uint32_t vbase = kbase + kKBytes;
        float sacc[2][2][4];  // [group][8-key block][fragment]
#pragma unroll
        for (int kg = 0; kg < 2; ++kg)
#pragma unroll
          for (int j = 0; j < 2; ++j) sacc[kg][j][0] = sacc[kg][j][1] = sacc[kg][j][2] = sacc[kg][j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int kg = 0; kg < 2; ++kg) {
            // matrices: (keys 0-7, chunk 2kk), (keys 8-15, chunk 2kk),
            //           (keys 0-7, chunk 2kk+1), (keys 8-15, chunk 2kk+1)
            uint32_t r[4];
            ldsm_x4(kbase + sw128(warp * 32 + kg * 16 + k_row, 2 * kk + k_chi), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t b0, b1;
              e4m3x4_to_f16x2(r[j], b0, b1);
              mma_16816_f16(sacc[kg][j & 1], qf[2 * kk + (j >> 1)], b0, b1);
            }
          }
        }
#pragma unroll
        for (int kg = 0; kg < 2; ++kg)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int32_t key = key0 + 16 * kg + 8 * j + 2 * tq + (e & 1);
              sacc[kg][j][e] = (key < n_slots) ? sacc[kg][j][e] * sl2[e >> 1] : -INFINITY;
            }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int kg = 0; kg < 2; ++kg)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            mx0 = fmax3(mx0, sacc[kg][j][0], sacc[kg][j][1]);
            mx1 = fmax3(mx1, sacc[kg][j][2], sacc[kg][j][3]);
          }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // Lazy rescale: a row's running max moves (and the accumulators are
        // rescaled) only when the tile's max exceeds it by more than 2^8, so
        // P <= 256 (exact enough in f16, and the sums stay far from overflow).
        // The final o / l and lse = m + log2(l) use whichever max the row kept.
        const bool up0 = mx0 > m0 + kLazyRescale, up1 = mx1 > m1 + kLazyRescale;  // m = -inf: up
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
          const float a0 = up0 ? fast_exp2(m0 - mn0) : 1.f, a1 = up1 ? fast_exp2(m1 - mn1) : 1.f;
          m0 = mn0;
          m1 = mn1;
          l0 *= a0;
          l1 *= a1;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            oacc[i][0] *= a0;
            oacc[i][1] *= a0;
            oacc[i][2] *= a1;
            oacc[i][3] *= a1;
          }
        }
#pragma unroll
        for (int kg = 0; kg < 2; ++kg) {
          float pr[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            pr[j][0] = fast_exp2(sacc[kg][j][0] - m0);
            pr[j][1] = fast_exp2(sacc[kg][j][1] - m0);
            pr[j][2] = fast_exp2(sacc[kg][j][2] - m1);
            pr[j][3] = fast_exp2(sacc[kg][j][3] - m1);
          }
          l0 += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
          l1 += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
          uint32_t pa[4];
          pa[0] = pack_f16x2(pr[0][0], pr[0][1]);
          pa[1] = pack_f16x2(pr[0][2], pr[0][3]);
          pa[2] = pack_f16x2(pr[1][0], pr[1][1]);
          pa[3] = pack_f16x2(pr[1][2], pr[1][3]);
          // O += P V over this group's 16 keys: transposed tile (warp * 32 +
          // 16 kg) / 64, its 16-key column chunk ((2 warp + kg) mod 4)
          const uint32_t vt = vbase + ((warp * 32 + kg * 16) / kVT) * (kD * kVT);
          const uint32_t vchunk = (2 * warp + kg) & 3;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t r[4];
            ldsm_x4(vt + sw64(32 * q4 + v_row, vchunk), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t b0, b1;
              e4m3x4_to_f16x2(r[j], b0, b1);
              mma_16816_f16(oacc[4 * q4 + j], pa, b0, b1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }

    // ------------------------------------------- merge the four warps ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    constexpr int kRowPad = kD + 8;
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    float *mo = reinterpret_cast<float *>(smem);
    float *ml = mo + kDecWarps * kGroup * kRowPad;
    if (tq == 0) {
      ml[warp * kGroup + gr] = ok ? m0 : -INFINITY;
      ml[warp * kGroup + gr + 8] = ok ? m1 : -INFINITY;
      ml[kDecWarps * kGroup + warp * kGroup + gr] = ok ? l0 : 0.f;
      ml[kDecWarps * kGroup + warp * kGroup + gr + 8] = ok ? l1 : 0.f;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    const float vs = p.v_scale[g];
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
      // the V scale turns code values back into values
      f[h] = (L > 0.f && mine != -INFINITY) ? fast_exp2(mine - M) / L * vs : 0.f;
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
#pragma unroll 4
    for (int i = tid; i < kGroup * kD; i += kDecWarps * 32) {
      const int r = i / kD, d = i % kD;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) acc += mo[(w * kGroup + r) * kRowPad + d];
      if (p.splits == 1)
        p.o[(row0 + r) * kD + d] = __float2bfloat16_rn(acc);
      else
        part_o(r, d) = acc;
    }
    if (warp == 0 && tq == 0 && p.splits > 1) {
      part_lse(gr) = Lr[0] > 0.f ? Mr[0] + __log2f(Lr[0]) : -INFINITY;
      part_lse(gr + 8) = Lr[1] > 0.f ? Mr[1] + __log2f(Lr[1]) : -INFINITY;
    }
  } else {
    for (int i = threadIdx.x; i < kGroup * kD; i += kDecWarps * 32) {
      if (p.splits == 1)
        p.o[(row0 + i / kD) * kD + i % kD] = __float2bfloat16_rn(0.f);
      else
        part_o(i / kD, i % kD) = 0.f;
    }
    if (threadIdx.x < kGroup && p.splits > 1) part_lse(threadIdx.x) = -INFINITY;
  }
}

cudaError_t launch_decode_e4m3(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                               cudaStream_t s) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(decode_e4m3_kernel), kSmem, 4);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, kHkv, p.batch);
  return launch_pdl(decode_e4m3_kernel, grid, dim3(kDecThreads), kSmem, s, p, tk, tv);
}

}  // namespace mg
