// attn_combine.cu -- merge split-KV partial attention results.
//
// Each split s of a row left o_s (already divided by its own softmax sum)
// and lse_s = m_s + log2(l_s) in the base-2 domain.  The exact softmax over
// the union of the splits is o = sum_s 2^(lse_s - L) o_s / sum_s 2^(lse_s - L)
// with L = max_s lse_s; splits that saw no key carry lse = -inf and drop out.
// A separate launch (no inter-CTA waiting).  One CTA of 16 warps per row:
// warp w takes splits w, w+16, ... and each lane four output dims; all of a
// warp's loads are issued together, each warp merges against its own max,
// and warp 0 rescales and adds the 16 warp results from shared memory.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {
constexpr int kCombineWarps = 16;
}

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  pdl_wait();  // the partials come from the previous kernel
  pdl_launch_dependents();
  __shared__ float4 red[kCombineWarps][32];
  __shared__ float den_w[kCombineWarps], max_w[kCombineWarps];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits;
  const float *lse = p.part_lse + static_cast<size_t>(row) * S;
  const float4 *po = reinterpret_cast<const float4 *>(p.part_o + static_cast<size_t>(row) * S * kD);

  // Every load of this warp goes out at once: its splits' lse and partial
  // rows (up to kPerWarp each); the warp merges them against its own max.
  constexpr int kPerWarp = (kDecMaxSplits + kCombineWarps - 1) / kCombineWarps;
  float ls[kPerWarp];
  float4 v[kPerWarp];
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const int s_ = warp + k * kCombineWarps;
    if (s_ < S) {
      ls[k] = __ldg(lse + s_);
      v[k] = __ldg(po + static_cast<size_t>(s_) * (kD / 4) + lane);
    } else {
      ls[k] = -INFINITY;
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) m = fmaxf(m, ls[k]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kPerWarp; ++k) {
      const float w = (ls[k] == -INFINITY) ? 0.f : fast_exp2(ls[k] - m);
      den += w;
      acc.x = fmaf(w, v[k].x, acc.x);
      acc.y = fmaf(w, v[k].y, acc.y);
      acc.z = fmaf(w, v[k].z, acc.z);
      acc.w = fmaf(w, v[k].w, acc.w);
    }
  }
  red[warp][lane] = acc;
  if (lane == 0) {
    den_w[warp] = den;
    max_w[warp] = m;
  }
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, max_w[w]);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float d = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) {
        const float f = (max_w[w] == -INFINITY) ? 0.f : fast_exp2(max_w[w] - M);
        const float4 b = red[w][lane];
        a.x = fmaf(f, b.x, a.x);
        a.y = fmaf(f, b.y, a.y);
        a.z = fmaf(f, b.z, a.z);
        a.w = fmaf(f, b.w, a.w);
        d = fmaf(f, den_w[w], d);
      }
    }
    const float inv = d > 0.f ? 1.f / d : 0.f;
    uint2 out;
    out.x = pack_bf16x2(a.x * inv, a.y * inv);
    out.y = pack_bf16x2(a.z * inv, a.w * inv);
    *reinterpret_cast<uint2 *>(p.o + static_cast<size_t>(row) * kD + 4 * lane) = out;
  }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(p.rows), dim3(kCombineWarps * 32), 0, s, p);
}

}  // namespace mg
