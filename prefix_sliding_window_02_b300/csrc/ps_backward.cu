// ps_backward.cu -- backward of the Prefix-Sliding prefill (dQ, dK, dV).
//
// The truncated-backprop trainer of "Prefix Sliding for efficient test-time
// scaling" (agihunt.info, paragraph on RL) back-propagates through the last
// 4W tokens of a rollout under the prefix-sliding mask.  Given the forward's
// inputs, its O and LSE, and dO, this computes per query row i and admitted
// key j (scores s = scale * q_hat . k_hat, P = exp(s - LSE)):
//     dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),  D_i = dO_i . O_i,
//     dQ_hat_i = scale sum_j dS_ij k_hat_j,  dK_hat_j = scale sum_i dS_ij q_hat_i,
// and pulls dQ_hat, dK_hat back through the rotation (the transpose of a
// rotation is the rotation by the negative angle; the bf16 rounding of q_hat
// and k_hat passes gradients straight through).
//
// Three kernels, all without atomics:
//  1. bwd_prep_kernel rotates Q and K exactly as the forward's pre-pass does
//     (same angles, same rounding) and forms D_i = dO_i . O_i.
//  2. bwd_dq_kernel: one CTA per (128-query tile, query head, batch row); it
//     walks the key tiles the forward visits and accumulates dQ in TMEM.
//  3. bwd_dkdv_kernel: one CTA per (128-key tile, KV head, batch row); it walks
//     the query tiles that can admit one of its keys, for every query head of
//     the group, and accumulates dK and dV in TMEM.
// Every product is a tcgen05 MMA (bf16 operands, fp32 accumulators in TMEM).
// Operands that are consumed along K use the 128-byte-swizzled K-major tiles a
// TMA box {64, 1, 128, 1} writes; the same tiles serve as MN-major B operands
// (rows along K) for the accumulating products, as V does in the forward.
// The probabilities and dS are written back into TMEM as bf16 and read as the
// tensor-memory A operand.
#include "ps_internal.h"
#include "ps_rope.cuh"
#include "ps_tc.cuh"
#include "ps_tiles.cuh"

namespace ps {
namespace bwd {

constexpr int kBM = 128, kBN = 128, kHD = 128;
constexpr int kHalf = kBM * 64 * 2;  // one 64-column swizzled half block: 16 KB
constexpr int kTile = 2 * kHalf;     // 128 x 128 bf16: 32 KB
constexpr uint32_t kIdescSS = tc::idesc_bf16(128, 128, false);  // both operands K-major
constexpr uint32_t kIdescTS = tc::idesc_bf16(128, 128, true);   // B MN-major
constexpr int kSmem = 6 * kTile + 2048 /*barriers, LSE and D rows*/ + 1024 /*alignment*/;

struct Params {
  CUtensorMap tmq;   // rotated Q  {D, Hq, S, B}
  CUtensorMap tmk;   // rotated K  {D, Hkv, S, B}
  CUtensorMap tmv;   // V          {D, Hkv, S, B}
  CUtensorMap tmdo;  // dO         {D, Hq, S, B}
  const float* lse;   // [B, Hq, S] natural log
  const float* dsum;  // [B, Hq, S] D_i = dO_i . O_i
  const int32_t* q_start;
  const int32_t* prefix_len;
  float* dq;  // [B, S, Hq, D]
  float* dk;  // [B, S, Hkv, D]
  float* dv;  // [B, S, Hkv, D]
  int32_t* status;
  int32_t S, hq, hkv, W, nq;
  float scale, scale_log2;
  RopeTurns turns;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Writes one thread's row of a 128-wide fp32 accumulator, scaled and rotated
// back by -pos when `rot` (dQ, dK), plainly otherwise (dV).  Every thread of
// the warp calls it (tcgen05.ld is warp-collective); only rows with `valid`
// store.
__device__ __forceinline__ void store_row(uint32_t taddr, float* dst, bool valid, float mul,
                                          bool rot, int32_t pos, const RopeTurns& turns) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {  // columns [32c, 32c+32) pair with [64+32c, 96+32c)
    uint32_t a[32], b[32];
    tc::ld32(taddr + c * 32, a);
    tc::ld32(taddr + 64 + c * 32, b);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float x = __uint_as_float(a[e]) * mul, y = __uint_as_float(b[e]) * mul;
      float rx = x, ry = y;
      if (rot) {
        float cs, sn;
        rope_cos_sin(pos, turns.f[c * 32 + e], cs, sn);
        rx = x * cs + y * sn;  // rotation by -angle
        ry = y * cs - x * sn;
      }
      a[e] = __float_as_uint(rx);
      b[e] = __float_as_uint(ry);
    }
    if (valid) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        *reinterpret_cast<uint4*>(dst + c * 32 + e) =
            make_uint4(a[e], a[e + 1], a[e + 2], a[e + 3]);
        *reinterpret_cast<uint4*>(dst + 64 + c * 32 + e) =
            make_uint4(b[e], b[e + 1], b[e + 2], b[e + 3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 1. pre-pass
// ---------------------------------------------------------------------------
struct PrepParams {
  const uint4* q;   // [B, S, Hq, D]
  const uint4* k;   // [B, S, Hkv, D]
  const uint4* o;   // [B, S, Hq, D] forward output
  const uint4* dout;
  uint4* qh;        // rotated
  uint4* kh;
  float* dsum;      // [B, Hq, S]
  const int32_t* q_start;
  int32_t B, S, hq, hkv;
  RopeTurns turns;
};

constexpr int kPrepRows = 4;

__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  constexpr int VEC = 16, HALFV = 8;
  __shared__ float2 cs[kPrepRows][64];
  grid_dependency_wait();
  allow_dependents();
  const int64_t n_rows = (int64_t)p.B * p.S;
  const int heads = p.hq + p.hkv;
  for (int64_t r0 = (int64_t)blockIdx.x * kPrepRows; r0 < n_rows;
       r0 += (int64_t)gridDim.x * kPrepRows) {
    {
      const int rr = threadIdx.x >> 6, i = threadIdx.x & 63;
      const int64_t r = r0 + rr;
      if (r < n_rows) {
        const int b = (int)(r / p.S);
        const int32_t pos = p.q_start[b] + (int32_t)(r % p.S);
        float c, sn;
        rope_cos_sin(pos, p.turns.f[i], c, sn);
        cs[rr][i] = make_float2(c, sn);
      }
    }
    __syncthreads();
    for (int it = threadIdx.x; it < kPrepRows * heads * 8; it += blockDim.x) {
      const int g = it & 7;
      const int hd = (it >> 3) % heads;
      const int rr = (it >> 3) / heads;
      const int64_t r = r0 + rr;
      if (r >= n_rows) continue;
      uint4 ra, rb;
      if (hd < p.hq) {
        const int64_t base = (r * p.hq + hd) * VEC + g;
        rotate8(p.q[base], p.q[base + HALFV], &cs[rr][8 * g], ra, rb);
        p.qh[base] = ra;
        p.qh[base + HALFV] = rb;
      } else {
        const int64_t base = (r * p.hkv + (hd - p.hq)) * VEC + g;
        rotate8(p.k[base], p.k[base + HALFV], &cs[rr][8 * g], ra, rb);
        p.kh[base] = ra;
        p.kh[base + HALFV] = rb;
      }
    }
    // D_i = dO_i . O_i: one warp per (row, query head), 4 elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int w = warp; w < kPrepRows * p.hq; w += blockDim.x / 32) {
      const int64_t r = r0 + w / p.hq;
      const int h = w % p.hq;
      if (r >= n_rows) continue;
      const uint2* o2 = reinterpret_cast<const uint2*>(p.o) + (r * p.hq + h) * 32 + lane;
      const uint2* d2 = reinterpret_cast<const uint2*>(p.dout) + (r * p.hq + h) * 32 + lane;
      const uint2 a = *o2, d = *d2;
      float acc = bf16lo(a.x) * bf16lo(d.x) + bf16hi(a.x) * bf16hi(d.x) +
                  bf16lo(a.y) * bf16lo(d.y) + bf16hi(a.y) * bf16hi(d.y);
      acc = warp_sum(acc);
      if (lane == 0) {
        const int b = (int)(r / p.S);
        p.dsum[((int64_t)b * p.hq + h) * p.S + (r % p.S)] = acc;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// 2. dQ: one CTA per (query tile, query head, batch row)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) bwd_dq_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + kTile;
  uint8_t* sK = smem + 2 * kTile;  // [2]
  uint8_t* sV = smem + 4 * kTile;  // [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * kTile);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_free = bars + 3;   // [2]: the dQ product that read the stage is done
  uint64_t* s_done = bars + 5;    // S and dP of the current key tile are in TMEM
  uint64_t* all_done = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = p.nq - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.hq / p.hkv);
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, false);
  const int32_t q0r = qt * kBM, q1r = min(p.S, q0r + kBM) - 1;
  const int64_t q0 = (int64_t)c0 + q0r, q1 = (int64_t)c0 + q1r;
  // key tiles that can hold an admitted pair: the prefix tiles, then the band
  const int32_t kc = keys_below(km, q1 + 1);
  const int32_t kP = keys_below(km, P);
  const int t1_end = (min(kP, kc) + kBN - 1) / kBN;
  const int32_t kw = keys_below(km, q0 - p.W + 1);
  const int t2_begin = max(t1_end, kw / kBN);
  const int t2_end = (kc + kBN - 1) / kBN;
  const int n_tiles = t1_end + max(0, t2_end - t2_begin);
  auto tile_at = [&](int it) { return it < t1_end ? it : t2_begin + (it - t1_end); };

  if (warp == 0) {
    tc::alloc(smem_u32(tmem_slot), 512);
    tc::relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tP = tmem + 128, tQ = tmem + 256;  // S | dP -> dS | dQ
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  grid_dependency_wait();

  const uint64_t pol = policy_evict_last();
  auto load_kv = [&](int stage, int kt) {
    mbar_arrive_expect_tx(&kv_full[stage], 2 * kTile);
    tma_load_4d(sK + stage * kTile, &p.tmk, &kv_full[stage], 0, hk, kt * kBN, b, pol);
    tma_load_4d(sK + stage * kTile + kHalf, &p.tmk, &kv_full[stage], 64, hk, kt * kBN, b, pol);
    tma_load_4d(sV + stage * kTile, &p.tmv, &kv_full[stage], 0, hk, kt * kBN, b, pol);
    tma_load_4d(sV + stage * kTile + kHalf, &p.tmv, &kv_full[stage], 64, hk, kt * kBN, b, pol);
  };
  const uint64_t dq_ = tc::sdesc_sw128(smem_u32(sQ), 16, 1024);
  const uint64_t ddo = tc::sdesc_sw128(smem_u32(sdO), 16, 1024);
  const uint64_t dk_ = tc::sdesc_sw128(smem_u32(sK), 16, 1024);
  const uint64_t dv_ = tc::sdesc_sw128(smem_u32(sV), 16, 1024);
  const uint64_t dkm = tc::sdesc_sw128(smem_u32(sK), kHalf, 1024);  // K as an MN-major B
  if (tid == 0 && n_tiles > 0) {
    prefetch_tmap(&p.tmq);
    prefetch_tmap(&p.tmk);
    prefetch_tmap(&p.tmv);
    prefetch_tmap(&p.tmdo);
    mbar_arrive_expect_tx(q_full, 2 * kTile);
    tma_load_4d(sQ, &p.tmq, q_full, 0, h, q0r, b, pol);
    tma_load_4d(sQ + kHalf, &p.tmq, q_full, 64, h, q0r, b, pol);
    tma_load_4d(sdO, &p.tmdo, q_full, 0, h, q0r, b, pol);
    tma_load_4d(sdO + kHalf, &p.tmdo, q_full, 64, h, q0r, b, pol);
    for (int i = 0; i < 2 && i < n_tiles; ++i) load_kv(i, tile_at(i));
  }

  const int row = tid;
  const int32_t qrow = min(q0r + row, p.S - 1);
  const int64_t qpos = q0 + row;
  const float lse2 = p.lse[((int64_t)b * p.hq + h) * p.S + qrow] * 1.4426950408889634f;
  const float drow = p.dsum[((int64_t)b * p.hq + h) * p.S + qrow];
  // admitted key indices of this row: [0, a1) and [b0, b1)
  const int32_t a1 = keys_below(km, min((int64_t)P, qpos + 1));
  const int32_t b0 = keys_below(km, max((int64_t)0, qpos - p.W + 1));
  const int32_t b1 = keys_below(km, qpos + 1);
  bool ok = true;
  for (int it = 0; it < n_tiles; ++it) {
    const int st = it & 1;
    const int kt = tile_at(it);
    const int32_t ka = kt * kBN;
    if (tid == 0) {
      bool w = (it > 0 || mbar_wait(q_full, 0)) && mbar_wait(&kv_full[st], (it >> 1) & 1);
      if (w) {
        tc::fence_after();
        const uint64_t bk = dk_ + (uint64_t)((st * kTile) >> 4), bv = dv_ + (uint64_t)((st * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tS, dq_ + off, bk + off, kIdescSS, kk > 0);   // S = Q K^T
          tc::mma_bf16(tP, ddo + off, bv + off, kIdescSS, kk > 0);   // dP = dO V^T
        }
      } else {
        ok = false;
      }
      tc::commit(smem_u32(s_done));
      // the stage two tiles back is free once its dQ product is done: refill it
      if (w && it >= 1 && it + 1 < n_tiles) {
        const int sp = (it + 1) & 1;
        if (mbar_wait(&kv_free[sp], ((it - 1) >> 1) & 1)) {
          fence_proxy_async_smem();
          load_kv(sp, tile_at(it + 1));
        } else {
          ok = false;
        }
      }
    }
    if (!mbar_wait(s_done, it & 1)) ok = false;
    __syncwarp();
    tc::fence_after();
    // dS = P (dP - D) over this row, 32 keys at a time, written as bf16 over dP
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t sv[32], pv[32];
      tc::ld32(tS + lane_off + c * 32, sv);
      tc::ld32(tP + lane_off + c * 32, pv);
      tc::wait_ld();
      uint32_t packed[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float ds2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int32_t kx = ka + c * 32 + e + u;
          const bool keep = (kx < a1) || (kx >= b0 && kx < b1);
          const float pr = keep ? ex2(__uint_as_float(sv[e + u]) * p.scale_log2 - lse2) : 0.f;
          ds2[u] = pr * (__uint_as_float(pv[e + u]) - drow);
        }
        packed[e / 2] = pack_bf16(ds2[0], ds2[1]);
      }
      // chunk c's 16 packed columns land on dP columns already read (16c < 32c + 32)
      uint32_t* pk = packed;
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
          "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tP + lane_off + c * 16),
          "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]),
          "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]),
          "r"(pk[14]), "r"(pk[15])
          : "memory");
    }
    tc::wait_st();
    tc::fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    if (tid == 0) {  // dQ += dS K
      tc::fence_after();
      const uint64_t bk = dkm + (uint64_t)((st * kTile) >> 4);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        tc::mma_bf16_ts(tQ, tP + kk * 8, bk + ((kk * 2048) >> 4), kIdescTS, it > 0 || kk > 0);
      tc::commit(smem_u32(&kv_free[st]));
    }
  }
  if (tid == 0) tc::commit(smem_u32(all_done));
  if (ok && n_tiles > 0 && !mbar_wait(all_done, 0)) ok = false;
  ok = __syncthreads_and(ok) != 0;
  if (ok && n_tiles > 0) {
    tc::fence_after();
    const bool valid = q0r + row <= q1r;
    store_row(tQ + lane_off, p.dq + (((int64_t)b * p.S + (valid ? q0r + row : 0)) * p.hq + h) * kHD,
              valid, p.scale, true, (int32_t)qpos, p.turns);
  } else if (!ok && tid == 0) {
    set_flag(p.status, PS_DEV_TIMEOUT);
  }
  tc::fence_before();
  __syncthreads();
  if (!ok) {  // let copies and products already issued land before releasing memory
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
    __syncthreads();
  }
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// 3. dK, dV: one CTA per (key tile, KV head, batch row)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) bwd_dkdv_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sQ = smem + 2 * kTile;   // [2]
  uint8_t* sdO = smem + 4 * kTile;  // [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * kTile);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;  // [2]
  uint64_t* q_free = bars + 3;  // [2]
  uint64_t* s_done = bars + 5;
  uint64_t* all_done = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  float* sl = reinterpret_cast<float*>(bars + 16);  // [2][128] LSE (log2) then D of a query tile

  const int tid = threadIdx.x, warp = tid >> 5;
  const int kt = (int)blockIdx.x;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int G = p.hq / p.hkv;
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const int32_t k0r = kt * kBN, k1r = min(p.S, k0r + kBN) - 1;
  const int64_t kpos0 = (int64_t)c0 + k0r, kpos1 = (int64_t)c0 + k1r;
  // query tiles that can admit one of these keys: from the tile holding the
  // first key onwards; prefix keys are seen by every later query, window keys
  // only by queries up to W - 1 positions later
  const int qt_begin = k0r / kBM;
  int qt_end = p.nq;
  if (kpos0 >= P) {
    const int64_t last = kpos1 + p.W - 1 - c0;  // last query row that sees key k1r
    qt_end = (int)min((int64_t)p.nq, last / kBM + 1);
  }
  const int n_q = max(0, qt_end - qt_begin);
  const int n_iter = n_q * G;  // (query tile, head of the group) pairs

  if (warp == 0) {
    tc::alloc(smem_u32(tmem_slot), 512);
    tc::relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  // S^T -> P^T | dP^T -> dS^T | dV | dK
  const uint32_t tS = tmem, tP = tmem + 128, tV = tmem + 256, tK = tmem + 384;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  grid_dependency_wait();

  const uint64_t pol = policy_evict_last();
  auto load_q = [&](int stage, int j) {  // pair j: query tile qt_begin + j / G, head hk*G + j % G
    const int qt = qt_begin + j / G, h = hk * G + j % G;
    mbar_arrive_expect_tx(&q_full[stage], 2 * kTile);
    tma_load_4d(sQ + stage * kTile, &p.tmq, &q_full[stage], 0, h, qt * kBM, b, pol);
    tma_load_4d(sQ + stage * kTile + kHalf, &p.tmq, &q_full[stage], 64, h, qt * kBM, b, pol);
    tma_load_4d(sdO + stage * kTile, &p.tmdo, &q_full[stage], 0, h, qt * kBM, b, pol);
    tma_load_4d(sdO + stage * kTile + kHalf, &p.tmdo, &q_full[stage], 64, h, qt * kBM, b, pol);
  };
  const uint64_t dk_ = tc::sdesc_sw128(smem_u32(sK), 16, 1024);
  const uint64_t dv_ = tc::sdesc_sw128(smem_u32(sV), 16, 1024);
  const uint64_t dq_ = tc::sdesc_sw128(smem_u32(sQ), 16, 1024);
  const uint64_t ddo = tc::sdesc_sw128(smem_u32(sdO), 16, 1024);
  const uint64_t dqm = tc::sdesc_sw128(smem_u32(sQ), kHalf, 1024);   // Q as an MN-major B
  const uint64_t ddom = tc::sdesc_sw128(smem_u32(sdO), kHalf, 1024); // dO as an MN-major B
  if (tid == 0 && n_iter > 0) {
    prefetch_tmap(&p.tmq);
    prefetch_tmap(&p.tmk);
    prefetch_tmap(&p.tmv);
    prefetch_tmap(&p.tmdo);
    mbar_arrive_expect_tx(kv_full, 2 * kTile);
    tma_load_4d(sK, &p.tmk, kv_full, 0, hk, k0r, b, pol);
    tma_load_4d(sK + kHalf, &p.tmk, kv_full, 64, hk, k0r, b, pol);
    tma_load_4d(sV, &p.tmv, kv_full, 0, hk, k0r, b, pol);
    tma_load_4d(sV + kHalf, &p.tmv, kv_full, 64, hk, k0r, b, pol);
    for (int i = 0; i < 2 && i < n_iter; ++i) load_q(i, i);
  }

  const int row = tid;  // key row of the tile
  const int64_t kpos = kpos0 + row;
  // queries that admit this key: positions [kpos, kend] (prefix keys: all later ones)
  const int64_t kend = kpos < P ? INT64_MAX : kpos + p.W - 1;
  bool ok = true;
  for (int it = 0; it < n_iter; ++it) {
    const int st = it & 1;
    const int qt = qt_begin + it / G, h = hk * G + it % G;
    const int32_t q0r = qt * kBM;
    const int64_t qp0 = (int64_t)c0 + q0r;
    // LSE (log2) and D of the tile's 128 queries, for every key row
    __syncthreads();  // the previous iteration's readers of sl are done
    {
      const int32_t qr = min(q0r + tid, p.S - 1);
      sl[tid] = p.lse[((int64_t)b * p.hq + h) * p.S + qr] * 1.4426950408889634f;
      sl[128 + tid] = p.dsum[((int64_t)b * p.hq + h) * p.S + qr];
    }
    if (tid == 0) {
      bool w = (it > 0 || mbar_wait(kv_full, 0)) && mbar_wait(&q_full[st], (it >> 1) & 1);
      if (w) {
        tc::fence_after();
        const uint64_t bq = dq_ + (uint64_t)((st * kTile) >> 4), bo = ddo + (uint64_t)((st * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tS, dk_ + off, bq + off, kIdescSS, kk > 0);   // S^T = K Q^T
          tc::mma_bf16(tP, dv_ + off, bo + off, kIdescSS, kk > 0);   // dP^T = V dO^T
        }
      } else {
        ok = false;
      }
      tc::commit(smem_u32(s_done));
      if (w && it >= 1 && it + 1 < n_iter) {
        const int sp = (it + 1) & 1;
        if (mbar_wait(&q_free[sp], ((it - 1) >> 1) & 1)) {
          fence_proxy_async_smem();
          load_q(sp, it + 1);
        } else {
          ok = false;
        }
      }
    }
    __syncthreads();  // sl is written
    if (!mbar_wait(s_done, it & 1)) ok = false;
    __syncwarp();
    tc::fence_after();
#pragma unroll
    for (int c = 0; c < kBM / 32; ++c) {
      uint32_t sv[32], pv[32];
      tc::ld32(tS + lane_off + c * 32, sv);
      tc::ld32(tP + lane_off + c * 32, pv);
      tc::wait_ld();
      uint32_t pk_p[16], pk_s[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float pr2[2], ds2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = c * 32 + e + u;  // query of the tile
          const int64_t qpos = qp0 + i;
          const bool keep = q0r + i < p.S && qpos >= kpos && qpos <= kend;
          const float pr = keep ? ex2(__uint_as_float(sv[e + u]) * p.scale_log2 - sl[i]) : 0.f;
          pr2[u] = pr;
          ds2[u] = pr * (__uint_as_float(pv[e + u]) - sl[128 + i]);
        }
        pk_p[e / 2] = pack_bf16(pr2[0], pr2[1]);
        pk_s[e / 2] = pack_bf16(ds2[0], ds2[1]);
      }
      uint32_t* a = pk_p;
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
          "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tS + lane_off + c * 16),
          "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
          "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]),
          "r"(a[15])
          : "memory");
      uint32_t* d = pk_s;
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
          "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tP + lane_off + c * 16),
          "r"(d[0]), "r"(d[1]), "r"(d[2]), "r"(d[3]), "r"(d[4]), "r"(d[5]), "r"(d[6]), "r"(d[7]),
          "r"(d[8]), "r"(d[9]), "r"(d[10]), "r"(d[11]), "r"(d[12]), "r"(d[13]), "r"(d[14]),
          "r"(d[15])
          : "memory");
    }
    tc::wait_st();
    tc::fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    if (tid == 0) {  // dV += P^T dO, dK += dS^T Q
      tc::fence_after();
      const uint64_t bo = ddom + (uint64_t)((st * kTile) >> 4), bq = dqm + (uint64_t)((st * kTile) >> 4);
#pragma unroll
      for (int kk = 0; kk < kBM / 16; ++kk) {
        tc::mma_bf16_ts(tV, tS + kk * 8, bo + ((kk * 2048) >> 4), kIdescTS, it > 0 || kk > 0);
        tc::mma_bf16_ts(tK, tP + kk * 8, bq + ((kk * 2048) >> 4), kIdescTS, it > 0 || kk > 0);
      }
      tc::commit(smem_u32(&q_free[st]));
    }
  }
  if (tid == 0) tc::commit(smem_u32(all_done));
  if (ok && n_iter > 0 && !mbar_wait(all_done, 0)) ok = false;
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
    tc::fence_after();
    const bool valid = k0r + row <= k1r;
    const int64_t base = (((int64_t)b * p.S + (valid ? k0r + row : 0)) * p.hkv + hk) * kHD;
    if (n_iter > 0) {
      store_row(tV + lane_off, p.dv + base, valid, 1.f, false, 0, p.turns);
      store_row(tK + lane_off, p.dk + base, valid, p.scale, true, (int32_t)kpos, p.turns);
    } else if (valid) {  // no query admits these keys: zero gradients
      for (int e = 0; e < kHD; e += 4) {
        *reinterpret_cast<float4*>(p.dv + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(p.dk + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else if (tid == 0) {
    set_flag(p.status, PS_DEV_TIMEOUT);
  }
  tc::fence_before();
  __syncthreads();
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
    __syncthreads();
  }
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, 512);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t q_off, k_off, d_off, total;
};

static Layout layout(int B, int S, int hq, int hkv, int D) {
  Layout L;
  L.q_off = 0;
  L.k_off = align256((size_t)B * S * hq * D * 2);
  L.d_off = L.k_off + align256((size_t)B * S * hkv * D * 2);
  L.total = L.d_off + align256((size_t)B * hq * S * 4);
  return L;
}

}  // namespace bwd
}  // namespace ps

using namespace ps;

extern "C" ps_status_t ps_prefill_backward_workspace_size(int32_t batch, int32_t seqlen,
                                                          int32_t n_q_heads, int32_t n_kv_heads,
                                                          int32_t head_dim, size_t* bytes) {
  if (!bytes || batch < 1 || seqlen < 1 || n_q_heads < 1 || n_kv_heads < 1 ||
      n_q_heads % n_kv_heads)
    return PS_ERR_INVALID_ARGUMENT;
  if (head_dim != bwd::kHD) return PS_ERR_UNSUPPORTED;
  *bytes = bwd::layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim).total;
  return PS_OK;
}

extern "C" ps_status_t ps_prefill_backward(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* d_out,
                                           int32_t batch, int32_t seqlen, const int32_t* q_start,
                                           const int32_t* prefix_len, int32_t window,
                                           int32_t n_q_heads, int32_t n_kv_heads,
                                           int32_t head_dim, float scale, double rope_theta,
                                           float* dq, float* dk, float* dv, void* workspace,
                                           size_t workspace_bytes, int32_t* status, void* stream) {
  if (!q || !k || !v || !out || !lse || !d_out || !q_start || !prefix_len || !dq || !dk || !dv)
    return PS_ERR_INVALID_ARGUMENT;
  if (batch < 1 || seqlen < 1 || window < 1 || n_q_heads < 1 || n_kv_heads < 1 ||
      n_q_heads % n_kv_heads || !(scale > 0.f) || !(rope_theta > 0.0))
    return PS_ERR_INVALID_ARGUMENT;
  if (head_dim != bwd::kHD) return PS_ERR_UNSUPPORTED;
  if (batch > 65535 || n_q_heads > 65535) return PS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(d_out) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return PS_ERR_ALIGNMENT;
  const bwd::Layout L = bwd::layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PS_ERR_WORKSPACE;
  if (workspace_bytes < L.total) return PS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;

  bwd::PrepParams g;
  g.q = static_cast<const uint4*>(q);
  g.k = static_cast<const uint4*>(k);
  g.o = static_cast<const uint4*>(out);
  g.dout = static_cast<const uint4*>(d_out);
  g.qh = reinterpret_cast<uint4*>(ws + L.q_off);
  g.kh = reinterpret_cast<uint4*>(ws + L.k_off);
  g.dsum = reinterpret_cast<float*>(ws + L.d_off);
  g.q_start = q_start;
  g.B = batch;
  g.S = seqlen;
  g.hq = n_q_heads;
  g.hkv = n_kv_heads;
  make_rope_turns(rope_theta, head_dim, &g.turns);
  {
    const int64_t groups = ((int64_t)batch * seqlen + bwd::kPrepRows - 1) / bwd::kPrepRows;
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
    const int64_t blocks = groups < cap ? groups : cap;
    if (launch_dependent(bwd::bwd_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, s, g) !=
        cudaSuccess)
      return PS_ERR_CUDA;
  }

  bwd::Params p;
  const uint64_t qd[4] = {(uint64_t)head_dim, (uint64_t)n_q_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t qs[3] = {(uint64_t)head_dim * 2, (uint64_t)n_q_heads * head_dim * 2,
                          (uint64_t)seqlen * n_q_heads * head_dim * 2};
  const uint64_t kd[4] = {(uint64_t)head_dim, (uint64_t)n_kv_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t ks[3] = {(uint64_t)head_dim * 2, (uint64_t)n_kv_heads * head_dim * 2,
                          (uint64_t)seqlen * n_kv_heads * head_dim * 2};
  const uint32_t box[4] = {64u, 1u, (uint32_t)bwd::kBM, 1u};
  const bool okm =
      encode_tmap(&p.tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ws + L.q_off, qd, qs, box,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_tmap(&p.tmk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ws + L.k_off, kd, ks, box,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_tmap(&p.tmv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, kd, ks, box,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_tmap(&p.tmdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, d_out, qd, qs, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  if (!okm) return PS_ERR_CUDA;
  p.lse = lse;
  p.dsum = reinterpret_cast<const float*>(ws + L.d_off);
  p.q_start = q_start;
  p.prefix_len = prefix_len;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.S = seqlen;
  p.hq = n_q_heads;
  p.hkv = n_kv_heads;
  p.W = window;
  p.nq = (seqlen + bwd::kBM - 1) / bwd::kBM;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  make_rope_turns(rope_theta, head_dim, &p.turns);
  if (cudaFuncSetAttribute(bwd::bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bwd::kSmem) != cudaSuccess ||
      cudaFuncSetAttribute(bwd::bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bwd::kSmem) != cudaSuccess)
    return PS_ERR_CUDA;
  if (launch_dependent(bwd::bwd_dq_kernel, dim3((unsigned)p.nq, (unsigned)n_q_heads, (unsigned)batch),
                       dim3(128), (size_t)bwd::kSmem, s, p) != cudaSuccess)
    return PS_ERR_CUDA;
  if (launch_dependent(bwd::bwd_dkdv_kernel,
                       dim3((unsigned)p.nq, (unsigned)n_kv_heads, (unsigned)batch), dim3(128),
                       (size_t)bwd::kSmem, s, p) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}
