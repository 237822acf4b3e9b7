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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline ps_status_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? PS_OK : PS_ERR_CUDA;
}

// Validates the host-visible fields of a cache descriptor.
ps_status_t check_cache(const ps_cache_desc* c);

}  // namespace ps
