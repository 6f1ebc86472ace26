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
//    swizzle, two 64-dim boxes per tile) into a 3-deep mbarrier ring.
//  * Four consumer warps take 16 keys each of every tile.  The 16 query heads
//    of the KV group form the M = 16 side of mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate) for both Q.K^T and P.V; the K fragments are loaded
//    with ldmatrix and, in a local layer, rotated in registers (dimension i
//    and i+64 land in the same thread).  Online softmax in base 2 with quad
//    shuffles; row sums stay per thread until the end.
//  * The four warps merge in shared memory; the CTA writes (o / l, lse) for
//    its split and the combine kernel merges the splits.
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

}  // namespace

__global__ void __launch_bounds__(kDecThreads, 2)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDecStages * kDecStageBytes);
  uint64_t *turns = bars + 2 * kDecStages;  // 64 entries

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool local = (p.kind == 0);

  const int32_t pq = p.pos[b];
  const bool bad = pq < 0 || pq >= p.max_len || (!local && pq >= p.slots);
  int32_t n_slots = 0;
  if (!bad) n_slots = local ? min(pq + 1, p.slots) : pq + 1;
  int32_t chunk = (n_slots + p.splits - 1) / p.splits;
  chunk = (chunk + kDecTile - 1) / kDecTile * kDecTile;
  const int32_t s0 = split * chunk;
  const int32_t s1 = min(s0 + chunk, n_slots);

  const size_t row0 = static_cast<size_t>(b) * kHq + g * kGroup;  // first query row of the group
  if (bad || s0 >= s1) {
    if (bad && split == 0 && threadIdx.x == 0) set_err(p.err, MG_DERR_POSITION);
    // no keys for this split: lse = -inf, o = 0
    for (int i = threadIdx.x; i < kGroup * kD; i += blockDim.x) {
      const size_t r = row0 + i / kD;
      p.part_o[(r * p.splits + split) * kD + (i % kD)] = 0.f;
      if (i % kD == 0) p.part_lse[r * p.splits + split] = -INFINITY;
    }
    return;
  }
  const int ntiles = (s1 - s0 + kDecTile - 1) / kDecTile;

  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * kDecStages;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kDecWarps);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < 64) turns[threadIdx.x] = p.rope.turn[threadIdx.x];
  __syncthreads();

  if (warp == kDecWarps) {
    // ------------------------------------------------ TMA producer warp ----
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const int32_t c2 = b * kHkv + g;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kDecStages;
        if (t >= kDecStages) {
          if (!mbar_wait(bar_empty + 8 * st, ((t / kDecStages) - 1) & 1, &abort_flag)) {
            abort_flag = 1;
            set_err(p.err, MG_DERR_TIMEOUT);
            break;
          }
        }
        const uint32_t dst = smem_base + st * kDecStageBytes;
        const uint32_t fb = bar_full + 8 * st;
        const int32_t row = s0 + t * kDecTile;
        mbar_arrive_expect_tx(fb, kDecStageBytes);
        tma_load_3d(dst, &tk, fb, 0, row, c2);
        tma_load_3d(dst + 8192, &tk, fb, 64, row, c2);
        tma_load_3d(dst + 16384, &tv, fb, 0, row, c2);
        tma_load_3d(dst + 24576, &tv, fb, 64, row, c2);
        ++issued;
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last stages issued.
      for (int t = max(0, issued - kDecStages); t < issued; ++t)
        (void)mbar_wait(bar_full + 8 * (t % kDecStages), (t / kDecStages) & 1, nullptr);
    }
    return;  // no CTA-wide barrier follows: consumers sync among themselves
  }

  // ------------------------------------------------------ consumer warps ----
  const int gr = lane >> 2;  // fragment row group (0..7)
  const int tq = lane & 3;   // thread in quad

  // Q fragments (A operand, 16 heads x 128 dims), rotated by R(p) when local.
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
    if (local) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {  // dims c..c+1 then c+8..c+9
          const int i = ks * 16 + 2 * tq + 8 * h8;
          float c0, s0f, c1, s1f;
          rope_cos_sin(pq, turns[i], c0, s0f);
          rope_cos_sin(pq, turns[i + 1], c1, s1f);
          rot_pair(qf[ks][2 * h8], qf[ks + 4][2 * h8], c0, s0f, c1, s1f);
          rot_pair(qf[ks][2 * h8 + 1], qf[ks + 4][2 * h8 + 1], c0, s0f, c1, s1f);
        }
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

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kDecStages;
    // ldmatrix / mma.sync are warp-collective: the whole warp goes on or stops
    if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (t / kDecStages) & 1, &abort_flag))) {
      abort_flag = 1;
      set_err(p.err, MG_DERR_TIMEOUT);
      ok = false;
      break;
    }
    const int32_t key0 = s0 + t * kDecTile + warp * 16;  // slot of this warp's first key
    if (key0 < s1) {
      const uint32_t kbase = smem_base + st * kDecStageBytes;
      const uint32_t vbase = kbase + 16384;
      float sacc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;

      // positions of this thread's two keys (n-tile 0 and 1), for RoPE
      int32_t kpos0 = 0, kpos1 = 0;
      if (local) {
        const int32_t sl0 = key0 + gr, sl1 = key0 + 8 + gr;
        kpos0 = pq - ((pq - sl0) & (kWindow - 1));
        kpos1 = pq - ((pq - sl1) & (kWindow - 1));
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t lo[4], hi[4];
        // dims 16ks.. (box 0) and 16ks+64.. (box 1): same row and chunk
        const uint32_t off = sw128(k_row, 2 * ks + k_chi);
        ldsm_x4(kbase + off, lo[0], lo[1], lo[2], lo[3]);
        ldsm_x4(kbase + 8192 + off, hi[0], hi[1], hi[2], hi[3]);
        if (local) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            const int i = ks * 16 + 2 * tq + 8 * h8;
            float c0, sn0, c1, sn1;
            rope_cos_sin(kpos0, turns[i], c0, sn0);
            rope_cos_sin(kpos0, turns[i + 1], c1, sn1);
            rot_pair(lo[h8], hi[h8], c0, sn0, c1, sn1);
            rope_cos_sin(kpos1, turns[i], c0, sn0);
            rope_cos_sin(kpos1, turns[i + 1], c1, sn1);
            rot_pair(lo[2 + h8], hi[2 + h8], c0, sn0, c1, sn1);
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
        const uint32_t addr =
            vbase + (chunk16 >> 3) * 8192 + sw128(v_row, chunk16 & 7);
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
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // every consumer is past its last read of the tiles before the stage
  // memory is reused for the merge
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
  float *mo = reinterpret_cast<float *>(smem);  // [4 warps][16 rows][128]
  float *ml = mo + kDecWarps * kGroup * kD;     // [4][16] m, then [4][16] l
  if (ok) {
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      const int c = nd * 8 + 2 * tq;
      mo[(warp * kGroup + gr) * kD + c] = oacc[nd][0];
      mo[(warp * kGroup + gr) * kD + c + 1] = oacc[nd][1];
      mo[(warp * kGroup + gr + 8) * kD + c] = oacc[nd][2];
      mo[(warp * kGroup + gr + 8) * kD + c + 1] = oacc[nd][3];
    }
    if (tq == 0) {
      ml[warp * kGroup + gr] = m0;
      ml[warp * kGroup + gr + 8] = m1;
      ml[kDecWarps * kGroup + warp * kGroup + gr] = l0;
      ml[kDecWarps * kGroup + warp * kGroup + gr + 8] = l1;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
  const int tid = threadIdx.x;  // 0..127
  for (int i = tid; i < kGroup * kD; i += kDecWarps * 32) {
    const int r = i / kD, d = i % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, ml[w * kGroup + r]);
    float L = 0.f, acc = 0.f;
    if (ok && M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = ml[w * kGroup + r];
        if (mw == -INFINITY) continue;
        const float f = fast_exp2(mw - M);
        L += f * ml[kDecWarps * kGroup + w * kGroup + r];
        acc += f * mo[(w * kGroup + r) * kD + d];
      }
    }
    const size_t row = row0 + r;
    const bool valid = ok && L > 0.f;
    p.part_o[(row * p.splits + split) * kD + d] = valid ? acc / L : 0.f;
    if (d == 0) p.part_lse[row * p.splits + split] = valid ? M + __log2f(L) : -INFINITY;
  }
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t s) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(decode_kernel), kDecSmem, 0);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, kHkv, p.batch);
  decode_kernel<<<grid, kDecThreads, kDecSmem, s>>>(p, tk, tv);
  return cudaGetLastError();
}

}  // namespace mg
