// ps_host.cu -- status strings, RoPE turn table, tensor-map encoding, cache checks.
#include <math.h>

#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "ps_internal.h"

namespace ps {

void make_rope_turns(double theta, int head_dim, RopeTurns* out) {
  const long double two_pi = 6.283185307179586476925286766559005768L;
  const int half = head_dim / 2;
  for (int i = 0; i < kMaxHalfDim; ++i) {
    if (i >= half) {
      out->f[i] = 0;
      continue;
    }
    long double inv_freq = powl((long double)theta, -2.0L * (long double)i / (long double)head_dim);
    long double turns = inv_freq / two_pi;  // < 1 for theta >= 1
    turns = turns - floorl(turns);
    out->f[i] = (unsigned long long)ldexpl(turns, 64);
  }
}

static std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};
static std::atomic<int32_t> g_drop_first_load{0};

WaitHooks wait_hooks() {
  WaitHooks h;
  h.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  h.drop_first_load = g_drop_first_load.load(std::memory_order_relaxed);
  return h;
}

void set_wait_hooks(uint64_t wait_ns, int32_t drop_first_load) {
  g_wait_ns.store(wait_ns, std::memory_order_relaxed);
  g_drop_first_load.store(drop_first_load, std::memory_order_relaxed);
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

SlotMap slot_map(const ps_cache_desc* c) {
  SlotMap m;
  m.slot_base = c->slot_base;
  m.block_table = c->block_table;
  m.total_slots = c->total_slots;
  m.capacity = c->capacity;
  m.block_size = c->block_table ? c->block_size : 0;
  m.blocks_per_seq = c->block_table ? c->blocks_per_seq : 0;
  return m;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

ps_status_t check_cache(const ps_cache_desc* c) {
  if (!c || !c->k_pool || !c->v_pool || !c->prefix_len) return PS_ERR_INVALID_ARGUMENT;
  if (c->block_table) {
    if (c->block_size < 16 || c->block_size % 16 || c->blocks_per_seq < 1 ||
        (int64_t)c->blocks_per_seq * c->block_size < (int64_t)c->capacity)
      return PS_ERR_INVALID_ARGUMENT;
  } else if (!c->slot_base) {
    return PS_ERR_INVALID_ARGUMENT;
  }
  if (c->nseq < 1 || c->n_kv_heads < 1 || c->window < 1 || c->prefix_max < 0 ||
      c->total_slots < 1 || c->total_slots > 0x7fffffffLL || !(c->rope_theta > 0.0))
    return PS_ERR_INVALID_ARGUMENT;
  if ((int64_t)c->capacity < (int64_t)c->prefix_max + c->window) return PS_ERR_INVALID_ARGUMENT;
  if (c->pe_mode != PS_PE_CONTINUE && c->pe_mode != PS_PE_RESET) return PS_ERR_INVALID_ARGUMENT;
  if (c->head_dim != 64 && c->head_dim != 128) return PS_ERR_UNSUPPORTED;
  if (!aligned16(c->k_pool) || !aligned16(c->v_pool)) return PS_ERR_ALIGNMENT;
  return PS_OK;
}

}  // namespace ps

extern "C" const char* ps_status_string(ps_status_t s) {
  switch (s) {
    case PS_OK: return "PS_OK";
    case PS_ERR_INVALID_ARGUMENT: return "PS_ERR_INVALID_ARGUMENT";
    case PS_ERR_UNSUPPORTED: return "PS_ERR_UNSUPPORTED";
    case PS_ERR_ALIGNMENT: return "PS_ERR_ALIGNMENT";
    case PS_ERR_WORKSPACE: return "PS_ERR_WORKSPACE";
    case PS_ERR_CUDA: return "PS_ERR_CUDA";
    case PS_ERR_DEVICE: return "PS_ERR_DEVICE";
  }
  return "PS_ERR_UNKNOWN";
}

extern "C" ps_status_t ps_check_device_status(const int32_t* status, int32_t* host_flags) {
  if (!status || !host_flags) return PS_ERR_INVALID_ARGUMENT;
  int32_t v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PS_ERR_CUDA;
  *host_flags = v;
  return v ? PS_ERR_DEVICE : PS_OK;
}

extern "C" ps_status_t ps_test_force_wait_timeout(int32_t enable, int64_t wait_limit_ns) {
  if (enable != 0 && enable != 1) return PS_ERR_INVALID_ARGUMENT;
  if (enable && (wait_limit_ns < 1000 || wait_limit_ns > (int64_t)ps::kWaitLimitNs))
    return PS_ERR_INVALID_ARGUMENT;
  ps::set_wait_hooks(enable ? (uint64_t)wait_limit_ns : ps::kWaitLimitNs, enable);
  return PS_OK;
}
