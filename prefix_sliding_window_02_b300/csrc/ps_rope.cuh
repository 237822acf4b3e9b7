// ps_rope.cuh -- the half-split RoPE rotation of one 16-byte group of bf16 pairs,
// shared by the prefill pre-pass, the prefill tile kernel (which rotates its
// query tiles in shared memory) and the backward pre-pass, so that all of them
// round the rotated Q and K to the same bf16 values.
#pragma once

#include "ps_common.cuh"

namespace ps {

// One rotation pair (x: element i of the first half, y: its partner i + D/2)
// by the angle with cosine c and sine s; explicit roundings, shared by every
// kernel that rotates keys so that they all store the same bf16 values.
__device__ __forceinline__ float rope_first(float x, float y, float c, float s) {
  return __fmaf_rn(x, c, -__fmul_rn(y, s));
}
__device__ __forceinline__ float rope_second(float x, float y, float c, float s) {
  return __fmaf_rn(y, c, __fmul_rn(x, s));
}

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
    raw[e] = pack_bf16(rope_first(x0, y0, t0.x, t0.y), rope_first(x1, y1, t1.x, t1.y));
    rbw[e] = pack_bf16(rope_second(x0, y0, t0.x, t0.y), rope_second(x1, y1, t1.x, t1.y));
  }
}

}  // namespace ps
