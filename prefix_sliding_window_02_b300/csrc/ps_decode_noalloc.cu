// ps_decode_noalloc.cu -- ps_decode with its scratch in a fixed device array.
//
// ps_decode needs a few MB of device scratch for its split-KV partial
// results, which its caller normally allocates (ps_decode_workspace_size).
// Some callers cannot allocate device memory at the point where they decode:
// code running while a caching allocator is locked or being torn down,
// callers that budget every allocation up front and forbid growth during
// generation, or plain C hosts that link this library without any allocator
// of their own.  ps_decode_noalloc serves them: its scratch lives in one
// file-scope __device__ array that every GPU which loads this library holds
// until the process exits.
#include <mutex>

#include <cudaTypedefs.h>

#include "ps_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB

__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

// Device address of g_decode_scratch on the current device.  In host code the
// array's name stands for a host-side shadow, not for device memory, so the
// address must come from the runtime with the device current.  It is looked
// up once per device and cached together with the device's current context:
// if that context is destroyed and re-created (cudaDeviceReset, or the
// primary context released and retained again), the module is loaded anew,
// the array may sit elsewhere, and the address is looked up again.
ps_status_t scratch_for_current_device(void** out) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PS_ERR_UNSUPPORTED;
  if (!g_ctx_current) return PS_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return PS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
    // first use on this device, or its context changed: the lookup also makes
    // the runtime's context current when none was
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PS_ERR_CUDA;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return PS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return PS_OK;
}

}  // namespace

extern "C" ps_status_t ps_decode_noalloc(const ps_cache_desc* cache, const void* q,
                                         const int32_t* pos, int32_t n_q_heads, float scale,
                                         void* out, float* lse, void* stream) {
  if (!cache) return PS_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  ps_status_t st = ps_decode_workspace_size(cache->nseq, n_q_heads, cache->n_kv_heads,
                                            cache->head_dim, &need);
  if (st != PS_OK) return st;
  if (need > kStaticScratchBytes) return PS_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != PS_OK) return st;
  // Nothing in the scratch has to start at zero: the partial kernel writes the
  // per-sequence tile offsets and every record before the combine reads them.
  return ps_decode(cache, q, pos, n_q_heads, scale, out, lse, scratch, kStaticScratchBytes,
                   stream);
}
