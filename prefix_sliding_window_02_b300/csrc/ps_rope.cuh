// ps_rope.cuh -- the half-split RoPE rotation of one 16-byte group of bf16 pairs,
// shared by the prefill pre-pass, the prefill tile kernel (which rotates its
// query tiles in shared memory) and the backward pre-pass, so that all of them
// round the rotated Q and K to the same bf16 values.
#pragma once

#include "ps_common.cuh"

namespace ps {

// Rotates 8 rotation pairs: elements 8g..8g+7 of the first half (a) with their
// partners 8g+64.. of the second half (b); cs holds (cos, sin) of each pair.
__device__ __forceinline__ void rotate8(const uint4& a, const uint4& b, const float2* cs,
                                        uint4& ra, uint4& rb) {
  const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
  const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b);
  uint32_t* raw = reinterpret_cast<uint32_t*>(&ra);
  uint32_t* rbw = reinterpret_cast<uint32_t*>(&rb);
  // explicit roundings (no contraction left to the compiler), so that every
  // kernel that rotates a row gets the same bf16 result
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t0 = cs[2 * e], t1 = cs[2 * e + 1];
    const float x0 = bf16lo(aw[e]), x1 = bf16hi(aw[e]);
    const float y0 = bf16lo(bw[e]), y1 = bf16hi(bw[e]);
    raw[e] = pack_bf16(__fmaf_rn(x0, t0.x, -__fmul_rn(y0, t0.y)),
                       __fmaf_rn(x1, t1.x, -__fmul_rn(y1, t1.y)));
    rbw[e] = pack_bf16(__fmaf_rn(y0, t0.x, __fmul_rn(x0, t0.y)),
                       __fmaf_rn(y1, t1.x, __fmul_rn(x1, t1.y)));
  }
}

}  // namespace ps
