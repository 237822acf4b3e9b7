// ps_internal.h -- host-side helpers shared by the libps translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ps_common.cuh"

namespace ps {

// f_i = theta^(-2i/D) / (2 pi) in 0.64 fixed point, for i < D/2 (long double on the host).
void make_rope_turns(double theta, int head_dim, RopeTurns* out);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
// Returns false if the driver entry point or the encode call fails.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

int device_sm_count();  // SM count of the current device (0 on failure)

// Settings of the wait-timeout test hook (ps_test_force_wait_timeout): the
// bounded-wait limit the kernels get, and whether CTA 0 skips its first K/V copy.
struct WaitHooks {
  uint64_t wait_ns;
  int32_t drop_first_load;
};
WaitHooks wait_hooks();
void set_wait_hooks(uint64_t wait_ns, int32_t drop_first_load);

// Launches `kernel` with programmatic stream serialisation: it may be scheduled
// before the previous kernel in `stream` completes (see grid_dependency_wait).
template <typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline ps_status_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? PS_OK : PS_ERR_CUDA;
}

// Logical-slot -> pool-row map of a cache descriptor (contiguous or paged).
SlotMap slot_map(const ps_cache_desc* c);

// Validates the host-visible fields of a cache descriptor.
ps_status_t check_cache(const ps_cache_desc* c);

}  // namespace ps
