// rope_stage.cu -- RoPE-rotated, position-ordered copies of a local layer's
// queries and window keys for the tensor-core verify / prefill kernel.
//
// A local layer applies RoPE ("Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳
// Muse Glimmer", section "长上下文仍然带来计算开销": global layers leave it
// out, so the local ones carry it) and keeps its keys in a 2048-slot ring.
// For a chunk starting at c0 this kernel writes, per sequence and KV head,
// the rows of positions c0-2048 .. c0+n-1 in position order:
//   ks[row] = R(pos) k_pos,  vs[row] = v_pos,  row = pos - c0 + 2048,
// taking positions < c0 from the ring (slot pos mod 2048) and the rest from
// the chunk's own k_new / v_new; rows of negative positions are zero.  The
// queries are rotated the same way: qs = R(pos) q.  Rotation is in fp32 with
// exactly reduced angles (see rope_cos_sin); each rotated value x is stored as
// two bf16 values, hi = bf16(x) (ks, qs) and lo = bf16(x - hi) (ks_lo,
// qs_lo), which the tensor-core kernel multiplies as hi.hi + lo.hi + hi.lo so
// that the scores keep the rotation's fp32 precision.
#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

namespace {

// Two fp32 values as bf16 pairs hi = bf16(v) and lo = bf16(v - hi).
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo(hi), b - bf16hi(hi));
}

// Rotate dims 8c..8c+7 (x) and their partners 8c+64.. (y) by position pos;
// the rotated values come back as hi parts in (x, y) and lo parts in
// (xl, yl).  tt holds the turns as [e][c] (frequency 8c + e at 8e + c), so
// that the 8 values of c that a warp's lanes take sit side by side.
__device__ __forceinline__ void rotate8(uint4 &x, uint4 &y, uint4 &xl, uint4 &yl, int32_t pos,
                                        int c, const uint64_t *tt) {
  uint32_t *l = reinterpret_cast<uint32_t *>(&x);
  uint32_t *h = reinterpret_cast<uint32_t *>(&y);
  uint32_t *ll = reinterpret_cast<uint32_t *>(&xl);
  uint32_t *hl = reinterpret_cast<uint32_t *>(&yl);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float c0, s0, c1, s1;
    rope_cos_sin(pos, tt[8 * (2 * e) + c], c0, s0);
    rope_cos_sin(pos, tt[8 * (2 * e + 1) + c], c1, s1);
    const float x0 = bf16lo(l[e]), x1 = bf16hi(l[e]);
    const float y0 = bf16lo(h[e]), y1 = bf16hi(h[e]);
    split2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1, l[e], ll[e]);
    split2(x0 * s0 + y0 * c0, x1 * s1 + y1 * c1, h[e], hl[e]);
  }
}

}  // namespace

__global__ void __launch_bounds__(256) rope_stage_kernel(const __grid_constant__ StageParams p) {
  // The turns in shared memory, transposed: a warp's lanes index them by
  // their own 8-dim chunk, which the kernel-parameter bank would serialise.
  __shared__ uint64_t tt[64];
  if (threadIdx.x < 64) tt[8 * (threadIdx.x & 7) + (threadIdx.x >> 3)] = p.rope.turn[threadIdx.x];
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n_kv = static_cast<int64_t>(p.batch) * kHkv * p.R * 8;
  const int64_t n_q = static_cast<int64_t>(p.batch) * p.n * kHq * 8;
  if (idx >= n_kv + n_q) return;
  const int c = static_cast<int>(idx & 7);  // dims 8c..8c+7 and 64+8c..64+8c+7
  if (idx < n_kv) {
    const int64_t row_id = idx >> 3;
    const int32_t r = static_cast<int32_t>(row_id % p.R);
    const int g = static_cast<int>((row_id / p.R) % kHkv);
    const int b = static_cast<int>(row_id / (static_cast<int64_t>(p.R) * kHkv));
    const int32_t c0 = p.pos0[b];
    if (c0 < 0 || static_cast<int64_t>(c0) + p.n > p.max_len) return;  // flagged by the attention kernel
    const int64_t pos = static_cast<int64_t>(c0) - kWindow + r;
    uint4 klo = make_uint4(0, 0, 0, 0), khi = klo, vlo = klo, vhi = klo, klo_l = klo, khi_l = klo;
    if (pos >= 0) {
      const __nv_bfloat16 *ksrc, *vsrc;
      if (pos < c0) {
        const size_t off = ((static_cast<size_t>(b) * kHkv + g) * kWindow + (pos % kWindow)) * kD;
        ksrc = p.k_cache + off;
        vsrc = p.v_cache + off;
      } else {
        const size_t off = ((static_cast<size_t>(b) * p.n + (pos - c0)) * kHkv + g) * kD;
        ksrc = p.k_new + off;
        vsrc = p.v_new + off;
      }
      klo = __ldg(reinterpret_cast<const uint4 *>(ksrc + 8 * c));
      khi = __ldg(reinterpret_cast<const uint4 *>(ksrc + 64 + 8 * c));
      vlo = __ldg(reinterpret_cast<const uint4 *>(vsrc + 8 * c));
      vhi = __ldg(reinterpret_cast<const uint4 *>(vsrc + 64 + 8 * c));
      rotate8(klo, khi, klo_l, khi_l, static_cast<int32_t>(pos), c, tt);
    }
    const size_t dst = ((static_cast<size_t>(b) * kHkv + g) * p.R + r) * kD;
    *reinterpret_cast<uint4 *>(p.ks + dst + 8 * c) = klo;
    *reinterpret_cast<uint4 *>(p.ks + dst + 64 + 8 * c) = khi;
    *reinterpret_cast<uint4 *>(p.ks_lo + dst + 8 * c) = klo_l;
    *reinterpret_cast<uint4 *>(p.ks_lo + dst + 64 + 8 * c) = khi_l;
    *reinterpret_cast<uint4 *>(p.vs + dst + 8 * c) = vlo;
    *reinterpret_cast<uint4 *>(p.vs + dst + 64 + 8 * c) = vhi;
  } else {
    const int64_t row_id = (idx - n_kv) >> 3;  // (b, t, h)
    const int h = static_cast<int>(row_id % kHq);
    const int32_t t = static_cast<int32_t>((row_id / kHq) % p.n);
    const int b = static_cast<int>(row_id / (static_cast<int64_t>(kHq) * p.n));
    const int32_t c0 = p.pos0[b];
    if (c0 < 0 || static_cast<int64_t>(c0) + p.n > p.max_len) return;
    const size_t off = ((static_cast<size_t>(b) * p.n + t) * kHq + h) * kD;
    uint4 lo = __ldg(reinterpret_cast<const uint4 *>(p.q + off + 8 * c));
    uint4 hi = __ldg(reinterpret_cast<const uint4 *>(p.q + off + 64 + 8 * c));
    uint4 lo_l, hi_l;
    rotate8(lo, hi, lo_l, hi_l, c0 + t, c, tt);
    *reinterpret_cast<uint4 *>(p.qs + off + 8 * c) = lo;
    *reinterpret_cast<uint4 *>(p.qs + off + 64 + 8 * c) = hi;
    *reinterpret_cast<uint4 *>(p.qs_lo + off + 8 * c) = lo_l;
    *reinterpret_cast<uint4 *>(p.qs_lo + off + 64 + 8 * c) = hi_l;
  }
}

cudaError_t launch_rope_stage(const StageParams &p, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(p.batch) * kHkv * p.R * 8 +
                        static_cast<int64_t>(p.batch) * p.n * kHq * 8;
  const int64_t blocks = (total + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_pdl(rope_stage_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, p);
}

}  // namespace mg
