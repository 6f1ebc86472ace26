// decode_noalloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// Some callers of this library have no way to obtain a workspace: a plugin
// running inside a host framework that owns every device buffer and hands
// plugins none, or a latency-critical serving loop that must never call
// cudaMalloc (it can stall the whole device) and keeps no spare buffer for
// this layer.  mg_attn_decode_noalloc gives them the split-KV decode without
// a workspace argument: its split partials live in a fixed array compiled
// into this library (kNoAllocScratchBytes per GPU that loads it, held until
// the process exits).
//
// The array is shared by every call on a device and keeps whatever the last
// call wrote.  Nothing in it needs to start at zero: each split writes its
// whole partial result before the combine step reads it.  Two calls whose
// work overlaps on the GPU (different streams, or one still running when the
// next starts elsewhere) use the same memory and race.
//
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and remembers it, with the
// context it belongs to; make that first call before any stream capture
// begins, and again the first call after a device reset.
#include <mutex>

#include "mg_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MG_NOALLOC_SCRATCH_BYTES;

// Device-side scratch for the split partials.  Host code must not use this
// name as a pointer: on the host it is only a stand-in for the symbol, so its
// device address is looked up below.
__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;

// The address is remembered together with the context it was looked up in:
// after a device reset the runtime creates a new primary context, loads the
// library's module again and the array gets a new address, so a change of
// context means looking it up again.
struct ScratchSlot {
  CUcontext ctx;
  void *ptr;
};
ScratchSlot g_scratch[64] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// Device address of the scratch array on the current device, looked up the
// first time a device (or a new context of it) is seen.  Returns nullptr on
// failure.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const CtxGetCurrentFn get_ctx = ctx_get_current();
  if (get_ctx == nullptr) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
  ScratchSlot &slot = g_scratch[dev];
  if (ctx == nullptr || ctx != slot.ctx || slot.ptr == nullptr) {
    // (the lookup also creates the device's primary context if there is none yet)
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    slot.ctx = ctx;
    slot.ptr = p;
  }
  return slot.ptr;
}

}  // namespace

extern "C" int mg_attn_decode_noalloc(const mg_layer *layer, const mg_cache *cache,
                                      const int32_t *d_pos, int32_t max_len, const void *q,
                                      void *o, uint32_t *d_err, void *stream) {
  if (layer == nullptr || cache == nullptr) return MG_ERR_INVALID;
  const size_t need = mg_workspace_bytes(MG_OP_DECODE, layer, cache->batch, 1, max_len);
  if (need == static_cast<size_t>(-1)) return MG_ERR_INVALID;
  if (need > kNoAllocScratchBytes) return MG_ERR_WORKSPACE;  // batch x splits too large
  void *scratch = scratch_on_current_device();
  if (scratch == nullptr) return MG_ERR_CUDA;
  return mg_attn_decode(layer, cache, d_pos, max_len, q, o, scratch, kNoAllocScratchBytes, d_err,
                        stream);
}
