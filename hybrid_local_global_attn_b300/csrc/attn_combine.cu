// attn_combine.cu -- merge split-KV partial attention results.
//
// Each split s of a row left o_s (already divided by its own softmax sum)
// and lse_s = m_s + log2(l_s) in the base-2 domain.  The exact softmax over
// the union of the splits is o = sum_s 2^(lse_s - L) o_s / sum_s 2^(lse_s - L)
// with L = max_s lse_s; splits that saw no key carry lse = -inf and drop out.
// A separate launch (no inter-CTA waiting); one CTA of 128 threads per row,
// thread d owns output dim d.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  const int row = blockIdx.x;
  const int d = threadIdx.x;
  const float *lse = p.part_lse + static_cast<size_t>(row) * p.splits;
  const float *po = p.part_o + static_cast<size_t>(row) * p.splits * kD;
  float L = -INFINITY;
  for (int s = 0; s < p.splits; ++s) L = fmaxf(L, __ldg(lse + s));
  float acc = 0.f, den = 0.f;
  if (L != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float ls = __ldg(lse + s);
      if (ls == -INFINITY) continue;
      const float w = exp2f(ls - L);
      den += w;
      acc = fmaf(w, __ldg(po + static_cast<size_t>(s) * kD + d), acc);
    }
  }
  const float out = den > 0.f ? acc / den : 0.f;
  p.o[static_cast<size_t>(row) * kD + d] = __float2bfloat16_rn(out);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  combine_kernel<<<p.rows, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mg
