// kv_append.cu -- write new K/V rows into a layer's cache, verbatim.
//
// Local layers keep a 2048-slot ring (slot = pos mod 2048, the oldest entry
// is reused), global layers a linear cache (slot = pos); see "Tomas Koutsky
// 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer", section
// "窄缓存为长上下文留出空间" (evict or cyclically reuse stale entries).
// Pure data movement: one thread moves one 16-byte chunk of K and of V.
// The same kernel commits a verified draft block: only the accepted prefix
// of each sequence is written ("第三招：D-Flash投机解码实现3倍提速",
// kongchang.com: the main model checks the drafted block in one pass and
// keeps what it accepts).
#include <cuda_fp8.h>

#include "mg_internal.h"
#include "mg_ptx.cuh"

namespace mg {

// e4m3 codes (round to nearest even, saturated) of 8 bf16 values times mul,
// in memory order.
__device__ __forceinline__ uint2 e4m3_pack8(uint4 raw, float mul) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * mul;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * mul;
    const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    out[i >> 1] |= (two & 0xFFFFu) << (16 * (i & 1));
  }
  return make_uint2(out[0], out[1]);
}

// Thread idx of sequence b moves one 16-byte chunk of one K row and one V row.
__device__ __forceinline__ void append_chunk(const AppendParams &p, int b, int64_t idx) {
  const int64_t total = static_cast<int64_t>(p.n) * (kHkv * 16);
  if (idx >= total) return;
  const int32_t t = static_cast<int32_t>(idx >> 5);  // token within the call
  const int g = static_cast<int>(idx >> 4) & 1;      // KV head
  const int c = static_cast<int>(idx & 15);          // 16-byte chunk of the row
  const int32_t pos0 = p.pos0[b];
  // Tokens of this sequence to write: all n, or the committed prefix.
  int32_t nb = p.n;
  bool skip = pos0 < 0;
  uint32_t why = MG_DERR_POSITION;
  if (p.count != nullptr) {
    nb = p.count[b];
    if (nb < 0 || nb > p.n) {
      skip = true;
      why = MG_DERR_COUNT;
    } else if (static_cast<int64_t>(pos0) + nb > 0x7fffffff) {
      skip = true;  // the next position would not fit an int32
    }
    if (idx == 0 && p.pos_next != nullptr) p.pos_next[b] = skip ? pos0 : pos0 + nb;
  }
  if (skip) {
    if (idx == 0) set_err(p.err, why);
    return;
  }
  if (t >= nb) return;  // rejected draft: never written
  // A ring keeps only the last `slots` tokens of this call; skipping the
  // earlier ones gives the same final state as appending one at a time and
  // avoids two writers racing for one slot.
  if (p.kind == 0 && t < nb - p.slots) return;
  const int64_t pos = static_cast<int64_t>(pos0) + t;
  int64_t slot;
  if (p.kind == 0) {
    slot = pos % p.slots;
  } else {
    if (pos >= p.slots) {
      set_err(p.err, MG_DERR_POSITION);
      return;
    }
    slot = pos;
  }
  const size_t src = ((static_cast<size_t>(b) * p.n + t) * kHkv + g) * kD + c * 8;
  if (p.dtype == MG_E4M3) {
    // FP8 global cache (linear): 8 dims of K -> 8 code bytes of the K row;
    // 8 dims of V -> one code byte in each of 8 rows of the transposed tile
    const uint4 kraw = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src));
    const uint4 vraw = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src));
    const uint2 kc = e4m3_pack8(kraw, p.k_mul[g]);
    const uint2 vc = e4m3_pack8(vraw, p.v_mul[g]);
    const size_t head = static_cast<size_t>(b) * kHkv + g;
    uint8_t *kdst = reinterpret_cast<uint8_t *>(p.k_cache) + (head * p.slots + slot) * kD + c * 8;
    *reinterpret_cast<uint2 *>(kdst) = kc;
    const int j = static_cast<int>(slot % 16);
    const int col = 16 * static_cast<int>((slot % 64) / 16) + 4 * ((j % 8) / 2) + 2 * (j / 8) + j % 2;
    uint8_t *vdst = reinterpret_cast<uint8_t *>(p.v_cache) +
                    (head * (p.slots / 64) + slot / 64) * (kD * 64) + static_cast<size_t>(c * 8) * 64 + col;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      vdst[i * 64] = static_cast<uint8_t>((i < 4 ? vc.x : vc.y) >> (8 * (i & 3)));
    return;
  }
  size_t dst;
  if (p.kind == 0) {
    dst = ((static_cast<size_t>(b) * kHkv + g) * p.slots + slot) * kD + c * 8;
  } else {
    int32_t row, outer;
    cache_coord(p.map, b, g, static_cast<int32_t>(slot), &row, &outer, c == 0 ? p.err : nullptr);
    dst = (static_cast<size_t>(outer) * p.map.rows + row) * kD + c * 8;
  }
  const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src));
  const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src));
  *reinterpret_cast<uint4 *>(p.k_cache + dst) = kv;
  *reinterpret_cast<uint4 *>(p.v_cache + dst) = vv;
}

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  pdl_wait();  // positions and rows may come from the previous kernel
  pdl_launch_dependents();
  append_chunk(p, blockIdx.y, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
}

// One commit into many layers' caches: blockIdx.z is the layer.  Only the
// first layer writes the next positions; every layer checks the counts.
__global__ void __launch_bounds__(256)
    kv_commit_layers_kernel(const __grid_constant__ CommitLayersParams cp) {
  pdl_wait();
  pdl_launch_dependents();
  const int l = blockIdx.z;
  AppendParams p = cp.common;
  const size_t off = static_cast<size_t>(l) * cp.layer_stride;
  p.k_new += off;
  p.v_new += off;
  p.k_cache = cp.k_cache[l];
  p.v_cache = cp.v_cache[l];
  p.slots = cp.slots[l];
  p.kind = cp.kind[l];
  p.map = cp.map[l];
  p.dtype = cp.dtype[l];
  p.k_mul[0] = cp.k_mul[l][0];
  p.k_mul[1] = cp.k_mul[l][1];
  p.v_mul[0] = cp.v_mul[l][0];
  p.v_mul[1] = cp.v_mul[l][1];
  if (l != 0) p.pos_next = nullptr;
  append_chunk(p, blockIdx.y, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
}

cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(p.n) * (kHkv * 16);
  const int64_t blocks = (total + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(p.batch));
  return launch_pdl(kv_append_kernel, grid, dim3(256), 0, s, p);
}

cudaError_t launch_kv_commit_layers(const CommitLayersParams &p, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(p.common.n) * (kHkv * 16);
  const int64_t blocks = (total + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(p.common.batch),
            static_cast<unsigned>(p.layers));
  return launch_pdl(kv_commit_layers_kernel, grid, dim3(256), 0, s, p);
}

}  // namespace mg
