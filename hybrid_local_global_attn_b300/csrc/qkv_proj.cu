// qkv_proj.cu -- the step before attention: each token's hidden state is
// projected to its query, key and value, and the key and value go straight
// into the layer's KV cache from the GEMM epilogue.
//
// What it computes ("深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？",
// section 01: hidden size 6656, 32 query heads and 2 KV heads of dimension
// 128): y = x W^T for x [M][6656] (M = batch x n tokens) and W [4608][6656],
// whose output features are the 32 query heads, then the 2 key heads, then
// the 2 value heads.  The bf16 rounding of y goes to q_out (and k_out /
// v_out when given); the key and value rows are also stored in the cache at
// their positions -- ring slot pos mod 2048 for a local layer, row pos of a
// linear or paged cache for a global one -- verbatim, as mg_kv_append would.
//
// Design (tcgen05, one 128 x 256 output tile at a time):
//  * warp 0: TMA producer, x and W in 64-wide K slices (128-byte swizzle)
//    through a 4-deep ring of 48 KB stages;
//  * warp 1: TMEM owner and single-thread MMA issuer, 4 M128 N256 K16 MMAs
//    per slice into one of two 256-column TMEM accumulators, so that a
//    tile's epilogue overlaps the next tile's main loop;
//  * warps 2-5: epilogue, thread = output row: TMEM -> registers -> bf16 ->
//    q / k / v rows and the cache rows.
//  * A persistent grid walks the tiles output-feature-fastest, so the CTAs
//    running at once share a few x panels and all of W in L2.
//  * With few tokens (decode) there are too few tiles for 148 SMs; the K
//    range is then split over CTAs that write fp32 partials, and a small
//    kernel sums them and runs the same epilogue.  That case is bound by
//    streaming W (61 MB) from HBM.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kKSteps = kHidden / kBK;          // 104
constexpr int kNTiles = kQkvFeatures / kBN;     // 18
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, 0, 0);
static_assert(kHidden % kBK == 0 && kQkvFeatures % kBN == 0, "tile shape");

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

struct Unit {
  int m_tile, n_tile, k0, k1;
};

__device__ __forceinline__ Unit unit_of(const QkvParams &p, int u) {
  const int mt = (p.M + kBM - 1) / kBM;
  Unit r;
  r.n_tile = u % kNTiles;
  const int rest = u / kNTiles;
  r.m_tile = rest % mt;
  const int split = rest / mt;
  r.k0 = split * p.ksteps;
  r.k1 = min(r.k0 + p.ksteps, kKSteps);
  return r;
}

// Final values of features f .. f+7 of token row m: q, k, v and the cache.
__device__ __forceinline__ void emit8(const QkvParams &p, int m, int f, const float (&v)[8]) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  if (f < kHq * kD) {
    *reinterpret_cast<uint4 *>(p.q_out + static_cast<size_t>(m) * (kHq * kD) + f) = w;
    return;
  }
  const bool is_k = f < (kHq + kHkv) * kD;
  const int fk = f - (is_k ? kHq * kD : (kHq + kHkv) * kD);  // within the 2 heads
  const int g = fk / kD, d = fk % kD;
  __nv_bfloat16 *out = is_k ? p.k_out : p.v_out;
  if (out != nullptr)
    *reinterpret_cast<uint4 *>(out + (static_cast<size_t>(m) * kHkv + g) * kD + d) = w;
  const int b = m / p.n, t = m % p.n;
  const int32_t p0 = p.pos0[b];
  if (p0 < 0 || p0 > 0x7fffffff - p.n) {  // the sequence's rows are not stored
    set_err(p.err, MG_DERR_POSITION);
    return;
  }
  const int32_t pos = p0 + t;
  __nv_bfloat16 *cache = is_k ? p.k_cache : p.v_cache;
  size_t row;
  if (p.kind == MG_LOCAL) {
    if (t < p.n - kWindow) return;  // a later token of this call takes the slot
    row = (static_cast<size_t>(b) * kHkv + g) * kWindow + (pos & (kWindow - 1));
  } else {
    if (pos >= p.slots) {
      set_err(p.err, MG_DERR_POSITION);
      return;
    }
    int32_t r, o;
    cache_coord(p.map, b, g, pos, &r, &o, p.err);
    row = static_cast<size_t>(o) * p.map.rows + r;
  }
  *reinterpret_cast<uint4 *>(cache + row * kD + d) = w;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const __grid_constant__ QkvParams p, const __grid_constant__ CUtensorMap tx,
                    const __grid_constant__ CUtensorMap tw) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sBar = sbase + kStages * kStageBytes;
  const uint32_t bar_full = sBar;                       // [kStages]
  const uint32_t bar_empty = bar_full + 8 * kStages;    // [kStages]
  const uint32_t bar_acc = bar_empty + 8 * kStages;     // [2] accumulator ready
  const uint32_t bar_accfree = bar_acc + 16;            // [2] accumulator drained (128)
  const uint32_t bar_done = bar_accfree + 16;           // every MMA retired
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (p.M + kBM - 1) / kBM;
  const int units = mt * kNTiles * p.splits;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_acc + 8 * i, 1);
      mbar_init(bar_accfree + 8 * i, 128);
    }
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tx);
    tma_prefetch_desc(&tw);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  pdl_wait();  // x (and the positions) come from earlier kernels
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------- producer ----
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit w = unit_of(p, u);
        for (int k = w.k0; k < w.k1; ++k, ++it) {
          const int st = it % kStages;
          if (it >= kStages &&
              !mbar_wait(bar_empty + 8 * st, ((it / kStages) - 1) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + st * kStageBytes;
          mbar_arrive_expect_tx(bar_full + 8 * st, kStageBytes);
          tma_load_2d(dst, &tx, bar_full + 8 * st, k * kBK, w.m_tile * kBM);
          tma_load_2d(dst + kABytes, &tw, bar_full + 8 * st, k * kBK, w.n_tile * kBN);
        }
      }
      if (!ok) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
      }
      // no copies may be in flight when the CTA retires
      for (int j = max(0, it - kStages); j < it; ++j)
        (void)mbar_wait(bar_full + 8 * (j % kStages), (j / kStages) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ----
    if (lane == 0) {
      int it = 0, lu = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++lu) {
        const Unit w = unit_of(p, u);
        const int ab = lu & 1;
        if (lu >= 2 && !mbar_wait(bar_accfree + 8 * ab, ((lu >> 1) - 1) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tbase + ab * kBN;
        for (int k = w.k0; k < w.k1; ++k, ++it) {
          const int st = it % kStages;
          if (!mbar_wait(bar_full + 8 * st, (it / kStages) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = sbase + st * kStageBytes, bb = a + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_ss(acc, smem_desc_sw128(a + 32 * kk, 16, 1024), smem_desc_sw128(bb + 32 * kk, 16, 1024),
                   kIdesc, (k > w.k0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * st);
        }
        if (!ok) break;
        mma_commit(bar_acc + 8 * ab);
      }
      if (!ok) {
        abort_flag = 1;
        set_err(p.err, MG_DERR_TIMEOUT);
      }
      mma_commit(bar_done);
      (void)mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // --------------------------------------------------------- epilogue ----
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = output row of the tile
    const uint32_t lane_bits = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    int lu = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++lu) {
      const Unit w = unit_of(p, u);
      const int ab = lu & 1;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_acc + 8 * ab, (lu >> 1) & 1, &abort_flag));
      if (!ok) break;  // warp-uniform; the MMA issuer stops on the abort flag
      tc_fence_after();
      const int m = w.m_tile * kBM + r;
      const int split = (u / kNTiles) / mt;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_bits + ab * kBN + 32 * c, v);
        tmem_wait_ld();
        if (m >= p.M) continue;
        const int f = w.n_tile * kBN + 32 * c;
        if (p.splits > 1) {
          float4 *dst = reinterpret_cast<float4 *>(
              p.part + (static_cast<size_t>(split) * p.M + m) * kQkvFeatures + f);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                 __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = __uint_as_float(v[8 * j + i]);
            emit8(p, m, f + 8 * j, e);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_accfree + 8 * ab);
    }
    if (!ok && lane == 0) set_err(p.err, MG_DERR_TIMEOUT);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Sum of the split partials of 8 features, then the epilogue.
__global__ void __launch_bounds__(256) qkv_reduce_kernel(const __grid_constant__ QkvParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t chunks = static_cast<int64_t>(p.M) * (kQkvFeatures / 8);
  if (i >= chunks) return;
  const int m = static_cast<int>(i / (kQkvFeatures / 8));
  const int f = static_cast<int>(i % (kQkvFeatures / 8)) * 8;
  float e[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < p.splits; ++s) {
    const float4 *src =
        reinterpret_cast<const float4 *>(p.part + (static_cast<size_t>(s) * p.M + m) * kQkvFeatures + f);
    const float4 a = src[0], b = src[1];
    e[0] += a.x; e[1] += a.y; e[2] += a.z; e[3] += a.w;
    e[4] += b.x; e[5] += b.y; e[6] += b.z; e[7] += b.w;
  }
  emit8(p, m, f, e);
}

int qkv_splits(int32_t M) {
  const int tiles = (M + kBM - 1) / kBM * kNTiles;
  if (tiles >= 74) return 1;
  return max(1, min(8, 148 / tiles));
}

cudaError_t launch_qkv(QkvParams p, const CUtensorMap &tx, const CUtensorMap &tw, cudaStream_t s) {
  if (p.M < 1 || p.splits < 1 || p.splits > 8) return cudaErrorInvalidValue;
  p.ksteps = (kKSteps + p.splits - 1) / p.splits;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(qkv_gemm_kernel), kSmem, 6);
  if (e != cudaSuccess) return e;
  const int units = (p.M + kBM - 1) / kBM * kNTiles * p.splits;
  e = launch_pdl(qkv_gemm_kernel, dim3(static_cast<unsigned>(min(units, 148))), dim3(kThreads), kSmem,
                 s, p, tx, tw);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t chunks = static_cast<int64_t>(p.M) * (kQkvFeatures / 8);
  return launch_pdl(qkv_reduce_kernel, dim3(static_cast<unsigned>((chunks + 255) / 256)), dim3(256), 0,
                    s, p);
}

}  // namespace mg
