// ps_math.cuh -- scalar and packed fp32 arithmetic used on the softmax paths
// of the prefill forward and backward kernels (sm_100+ instructions).
#pragma once

namespace ps {

// 2^x with the hardware approximation (flushes subnormals).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32x2 arithmetic and the three-input max of sm_100+: two elements
// (or two new candidates) per instruction on the softmax critical path.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Bits [lo, hi) of a 32-bit word (0 <= lo, hi <= 32; none when hi <= lo).
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  return (uint32_t)((1ull << hi) - 1) & ~(uint32_t)((1ull << lo) - 1);
}

// One bit per column c0 .. c0 + 31: set iff the column lies in [0, a1) or in
// [b0, b1).  A row's keep-mask is built once per tile, so the element mask of
// a partial tile costs a bit test and a select per element.
__device__ __forceinline__ uint32_t keep_bits(int c0, int32_t a1, int32_t b0, int32_t b1) {
  auto clamp32 = [](int32_t x) { return x < 0 ? 0 : (x > 32 ? 32 : x); };
  return bit_range(0, clamp32(a1 - c0)) | bit_range(clamp32(b0 - c0), clamp32(b1 - c0));
}

// d = a * b on two lanes at once.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

}  // namespace ps
