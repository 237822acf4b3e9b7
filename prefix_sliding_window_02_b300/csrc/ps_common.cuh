// ps_common.cuh -- device helpers shared by the libps kernels (sm_103a).
//
// RoPE angle: pos * theta^(-2i/D) radians is reduced modulo one turn exactly
// in 64-bit fixed point.  The host stores f_i = theta^(-2i/D) / (2 pi) as a
// 0.64 fixed-point fraction F_i; the device forms pos * F_i mod 2^64 (the
// fractional turn count of the angle), takes it as a signed fraction in
// [-1/2, 1/2) and calls sincospif.  No float64 arithmetic runs on the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ps.h"

namespace ps {

constexpr int kMaxHalfDim = 64;  // head_dim <= 128

struct RopeTurns {
  unsigned long long f[kMaxHalfDim];  // f_i * 2^64, i < D/2
};

__device__ __forceinline__ void rope_cos_sin(int32_t pos, unsigned long long F, float& c,
                                             float& s) {
  unsigned long long t = (unsigned long long)(uint32_t)pos * F;  // turns * 2^64 mod 2^64
  int32_t hi = (int32_t)(t >> 32);                                // signed turns * 2^32
  float x = (float)hi * 0x1p-31f;                                 // 2 * turns in [-1, 1)
  sincospif(x, &s, &c);
}

// Programmatic dependent launch.  The kernels of one call sequence are launched
// so that a kernel may be scheduled while the previous kernel in the stream is
// still running; each calls grid_dependency_wait() before it reads or writes
// any memory that earlier stream work touches (the wait returns once every
// earlier kernel has completed and its writes are visible; without the launch
// attribute it returns at once), and allow_dependents() to let the next kernel
// be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_flag(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- smem ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after limit_ns of wall time and returns false.  The
// kernels take the limit from their launch parameters (kWaitLimitNs unless a
// test shortens it, see ps_test_force_wait_timeout).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait shared by the roles of a warp-specialised CTA: it also gives up
// as soon as another role has given up (*abort set), and sets *abort itself
// when the time limit passes.
__device__ __forceinline__ bool mbar_wait_abort(uint64_t* bar, uint32_t parity,
                                                volatile int32_t* abort,
                                                uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

// ----------------------------------------------------------------- TMA ----
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(policy)
      : "memory");
}

// Plain (untiled) bulk copy global -> shared, completing on `bar`; both
// addresses 16-byte aligned, `bytes` a multiple of 16.
// Tiled store of a shared-memory box to global memory (bulk-group completion).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* m, const void* src, int32_t c0,
                                             int32_t c1, int32_t c2, int32_t c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(src)), "r"(c0), "r"(c1),
               "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------ warp reductions ----
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Pool row of a sequence's logical slot: contiguous from slot_base[s], or
// through a block table (paged cache).
struct SlotMap {
  const int64_t* slot_base;    // contiguous layout (block_table == nullptr)
  const int32_t* block_table;  // [nseq][blocks_per_seq] or nullptr
  int64_t total_slots;
  int32_t capacity, block_size, blocks_per_seq;

  // contiguous layout: the sequence's rows lie inside the pool
  __device__ __forceinline__ bool seq_ok(int s) const {
    if (block_table) return true;
    const int64_t sb = slot_base[s];
    return sb >= 0 && sb + capacity <= total_slots;
  }
  // row of logical slot `slot`, or -1 if its block lies outside the pool
  __device__ __forceinline__ int64_t row(int s, int32_t slot) const {
    if (!block_table) return slot_base[s] + slot;
    const int32_t blk = block_table[(int64_t)s * blocks_per_seq + slot / block_size];
    if (blk < 0 || (int64_t)(blk + 1) * block_size > total_slots) return -1;
    return (int64_t)blk * block_size + slot % block_size;
  }
};

// Ring slot of an absolute position (prefix slots fixed, window slots rotate).
__device__ __forceinline__ int32_t ring_slot(int32_t pos, int32_t P, int32_t W) {
  return pos < P ? pos : P + (pos - P) % W;
}

}  // namespace ps
