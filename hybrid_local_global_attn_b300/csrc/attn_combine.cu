// attn_combine.cu -- merge split-KV partial attention results.
//
// Each split s of a row left o_s (already divided by its own softmax sum)
// and lse_s = m_s + log2(l_s) in the base-2 domain.  The exact softmax over
// the union of the splits is o = sum_s 2^(lse_s - L) o_s / sum_s 2^(lse_s - L)
// with L = max_s lse_s; splits that saw no key carry lse = -inf and drop out.
// A separate launch (no inter-CTA waiting).  Few rows, many splits (global
// decode): one CTA of 16 warps per (row, quarter of the 128 dims): warp w
// takes splits w, w+16, ... with one dim per lane; all of a warp's loads are
// issued together, each warp merges against its own max, and warp 0
// rescales and adds the 16 warp results.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {
constexpr int kCombineWarps = 16;
constexpr int kCombineParts = kD / 32;  // CTAs per row, 32 dims each
}

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  // MG_OVERLAP_NEXT: the next kernel may begin at once
  if (p.overlap) pdl_launch_dependents();
  pdl_wait();  // the partials come from the previous kernel
  if (!p.overlap) pdl_launch_dependents();
  __shared__ float red[kCombineWarps][32];
  __shared__ float den_w[kCombineWarps], max_w[kCombineWarps];
  const int row = blockIdx.x / kCombineParts;
  const int d = (blockIdx.x % kCombineParts) * 32 + (threadIdx.x & 31);
  const int warp = threadIdx.x >> 5;
  const int S = p.splits;
  const float *lse = p.part_lse + static_cast<size_t>(row) * S;
  const float *po = p.part_o + static_cast<size_t>(row) * S * kD + d;

  constexpr int kPerWarp = (kDecMaxSplits + kCombineWarps - 1) / kCombineWarps;
  float ls[kPerWarp], v[kPerWarp];
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const int s_ = warp + k * kCombineWarps;
    ls[k] = (s_ < S) ? __ldg(lse + s_) : -INFINITY;
    v[k] = (s_ < S) ? __ldg(po + static_cast<size_t>(s_) * kD) : 0.f;
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) m = fmaxf(m, ls[k]);
  float acc = 0.f, den = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kPerWarp; ++k) {
      const float w = (ls[k] == -INFINITY) ? 0.f : fast_exp2(ls[k] - m);
      den += w;
      acc = fmaf(w, v[k], acc);
    }
  }
  red[warp][threadIdx.x & 31] = acc;
  if ((threadIdx.x & 31) == 0) {
    den_w[warp] = den;
    max_w[warp] = m;
  }
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, max_w[w]);
    float a = 0.f, dd = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) {
        const float f = (max_w[w] == -INFINITY) ? 0.f : fast_exp2(max_w[w] - M);
        a = fmaf(f, red[w][threadIdx.x], a);
        dd = fmaf(f, den_w[w], dd);
      }
    }
    p.o[static_cast<size_t>(row) * kD + d] = __float2bfloat16_rn(dd > 0.f ? a / dd : 0.f);
  }
}

// Many rows, few splits (verify): one CTA per row, thread d = output dim d.
// The splits go in chunks of kRowChunk whose loads are all in flight; the
// chunk maxima rescale the running sums (online log-sum-exp).  The chunk is
// picked from the split count so that a row takes one L2 round trip, while
// the registers stay few enough for many row CTAs to be resident when the
// partials land: 16 (48 registers), 20, or 40 (a 16-token block at batch 1
// gets 148 / (2 KV heads x 2 query blocks) = 37 splits; 96 registers, 5 CTAs
// per SM, all 512 of its rows resident).  Against chunks of 16 for every
// count, one round instead of three made global verify at batch 1 3 % faster
// and a 49-split decode 10 %; below 17 splits the larger chunks only cost
// residency.
constexpr int kRowSplitsMax = 64;  // above this the wide kernel is used
template <int kRowChunk>
__global__ void __launch_bounds__(kD) combine_rows_kernel(const CombineParams p) {
  // MG_OVERLAP_NEXT: the next kernel may begin at once
  if (p.overlap) pdl_launch_dependents();
  pdl_wait();  // the partials come from the previous kernel
  if (!p.overlap) pdl_launch_dependents();
  const int row = blockIdx.x, d = threadIdx.x;
  const int S = p.splits;
  const float *lse = p.part_lse + static_cast<size_t>(row) * S;
  const float *po = p.part_o + static_cast<size_t>(row) * S * kD + d;
  float m = -INFINITY, den = 0.f, acc = 0.f;
  for (int s0 = 0; s0 < S; s0 += kRowChunk) {
    float ls[kRowChunk], v[kRowChunk];
#pragma unroll
    for (int k = 0; k < kRowChunk; ++k) {
      const int s_ = s0 + k;
      ls[k] = (s_ < S) ? __ldg(lse + s_) : -INFINITY;
      v[k] = (s_ < S) ? __ldg(po + static_cast<size_t>(s_) * kD) : 0.f;
    }
    float mc = -INFINITY;
#pragma unroll
    for (int k = 0; k < kRowChunk; ++k) mc = fmaxf(mc, ls[k]);
    if (mc == -INFINITY) continue;  // nothing in this chunk
    const float mn = fmaxf(m, mc);
    const float f = (m == -INFINITY) ? 0.f : fast_exp2(m - mn);
    den *= f;
    acc *= f;
    m = mn;
#pragma unroll
    for (int k = 0; k < kRowChunk; ++k) {
      const float w = (ls[k] == -INFINITY) ? 0.f : fast_exp2(ls[k] - m);
      den += w;
      acc = fmaf(w, v[k], acc);
    }
  }
  p.o[static_cast<size_t>(row) * kD + d] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.splits <= 16) return launch_pdl(combine_rows_kernel<16>, dim3(p.rows), dim3(kD), 0, s, p);
  if (p.splits <= 20) return launch_pdl(combine_rows_kernel<20>, dim3(p.rows), dim3(kD), 0, s, p);
  if (p.splits <= kRowSplitsMax)
    return launch_pdl(combine_rows_kernel<40>, dim3(p.rows), dim3(kD), 0, s, p);
  return launch_pdl(combine_kernel, dim3(p.rows * kCombineParts), dim3(kCombineWarps * 32), 0, s,
                    p);
}

}  // namespace mg
