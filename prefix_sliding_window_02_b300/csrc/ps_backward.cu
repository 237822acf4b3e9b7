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
// Two launches, no atomics:
//  1. bwd_prep_kernel rotates Q and K exactly as the forward's pre-pass does
//     (same angles, same rounding) and stores, per (head, query row), the pair
//     {LSE * log2(e), D_i = dO_i . O_i}.
//  2. bwd_kernel runs two kinds of CTA in one grid:
//       dK/dV CTAs, one per (128-key tile, KV head, batch row): the key tile's
//         K and V stay in shared memory while 64-query sub-tiles of Q and dO of
//         every query head of the group stream past;
//       dQ CTAs, one per (128-query tile, query head, batch row): Q and dO stay
//         while 64-key sub-tiles of K and V stream past (the forward's tiles).
//     Both recompute S and dP, so each (query, key) tile pair costs 7 products
//     instead of the 5 of a single pass that adds dQ with atomics.
//
// CTA roles (320 threads): warps 0-7 turn S and dP into P and dS (two warps
// per TMEM lane quadrant, each on 32 of the sub-tile's 64 columns), warp 8
// issues the TMA copies, warp 9 issues the tcgen05 MMAs.  TMEM (512 columns):
// two sub-tile buffers S_b | dP_b (64 + 64 columns each), then the fp32
// accumulators (dV | dK, or dQ).  P and dS are written back over S and dP as
// bf16 pairs and read from TMEM as the A operand of the accumulating products.
// The issuer runs one sub-tile ahead: S, dP of sub-tile i+1 are issued before
// it waits for dS of sub-tile i, so the tensor cores work while the softmax
// warps do.  Tensor-core instructions of one thread execute in issue order,
// which lets S, dP of sub-tile i+2 overwrite the buffer whose P and dS the
// products of sub-tile i have just read.
#include "ps_internal.h"
#include "ps_math.cuh"
#include "ps_rope.cuh"
#include "ps_tc.cuh"
#include "ps_tiles.cuh"

namespace ps {
namespace bwd {

constexpr int kBM = 128;                 // rows of the resident tile
constexpr int kBC = 64;                  // rows of a streamed sub-tile
constexpr int kHD = 128;                 // head dim
constexpr int kHalfR = kBM * 128;        // one 64-column swizzled half of a resident tile: 16 KB
constexpr int kHalfC = kBC * 128;        // the same for a sub-tile: 8 KB
constexpr int kTileR = 2 * kHalfR;       // 32 KB
constexpr int kTileC = 2 * kHalfC;       // 16 KB
constexpr int kSt = 4;                   // sub-tile stages in flight
constexpr int kStage = 2 * kTileC;       // two sub-tile operands per stage
constexpr int kLdBytes = kBC * 8;        // {LSE*log2e, D} pairs of one query sub-tile
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kSmem = 2 * kTileR + kSt * kStage + kSt * kLdBytes + 1024 /*barriers*/ +
                      1024 /*alignment*/;
constexpr uint32_t kIdescSub = tc::idesc_bf16(128, kBC, false);  // S, dP: N = 64, K-major B
constexpr uint32_t kIdescAcc = tc::idesc_bf16(128, kHD, true);   // accumulations: B MN-major
constexpr uint32_t kTAcc = 256;                                  // accumulator columns

struct Params {
  CUtensorMap tmq_r, tmq_c;    // rotated Q {D, Hq, S, B}: 128-row and 64-row boxes
  CUtensorMap tmdo_r, tmdo_c;  // dO
  CUtensorMap tmk_r, tmk_c;    // rotated K {D, Hkv, S, B}
  CUtensorMap tmv_r, tmv_c;    // V
  const float2* ld;            // [B, Hq, s_pad] {LSE * log2(e), D}; rows >= S are zero
  const int32_t* q_start;
  const int32_t* prefix_len;
  float* dq;  // [B, S, Hq, D]
  float* dk;  // [B, S, Hkv, D]
  float* dv;  // [B, S, Hkv, D]
  int32_t* status;
  int32_t S, s_pad, hq, hkv, W, B;
  int32_t nq;       // 128-row query tiles
  int32_t n_dkdv;   // CTAs of the dK/dV kind (the first ones of the grid)
  float scale, scale_log2;
  RopeTurns turns;
};

struct Bars {
  uint64_t res_full;                       // the resident tiles have landed
  uint64_t st_full[kSt], st_empty[kSt];    // sub-tile stages
  uint64_t s_full[2], ds_ready[2];         // TMEM sub-tile buffers
  uint64_t done;                           // every accumulation has completed
  uint32_t tmem_slot;
  int32_t abort;
};

// TMEM column of the K16 step kk (16 sub-tile columns) of the bf16 pairs a
// softmax warp pair writes over a 64-column buffer: the warp on columns
// [32h, 32h+32) packs them into [32h, 32h+16).
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 1) * 32 + (kk & 1) * 8; }

// Writes 32 columns (chunk c: [32c, 32c+32) paired with [64+32c, 96+32c)) of
// one thread's row of a 128-wide fp32 accumulator, scaled and rotated back by
// -pos when `rot` (dQ, dK), plainly otherwise (dV).  Every thread of the warp
// calls it (tcgen05.ld is warp-collective); only rows with `valid` store.
__device__ __forceinline__ void store_chunk(uint32_t taddr, float* dst, int c, bool valid, float mul,
                                            bool rot, int32_t pos, const RopeTurns& turns) {
  uint32_t a[32], b[32];
  tc::ld32(taddr + c * 32, a);
  tc::ld32(taddr + 64 + c * 32, b);
  tc::wait_ld();
  if (!valid) return;
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
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    *reinterpret_cast<uint4*>(dst + c * 32 + e) = make_uint4(a[e], a[e + 1], a[e + 2], a[e + 3]);
    *reinterpret_cast<uint4*>(dst + 64 + c * 32 + e) =
        make_uint4(b[e], b[e + 1], b[e + 2], b[e + 3]);
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
  const float* lse; // [B, Hq, S] natural log
  uint4* qh;        // rotated
  uint4* kh;
  float2* ld;       // [B, Hq, s_pad]
  const int32_t* q_start;
  int32_t B, S, s_pad, hq, hkv;
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
        const int s = (int)(r % p.S);
        const float l2 = p.lse[((int64_t)b * p.hq + h) * p.S + s] * 1.4426950408889634f;
        p.ld[((int64_t)b * p.hq + h) * p.s_pad + s] = make_float2(l2, acc);
      }
    }
    __syncthreads();
  }
  // padding rows [S, s_pad) of every (batch row, head): zero
  const int pad = p.s_pad - p.S;
  const int64_t n_pad = (int64_t)p.B * p.hq * pad;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n_pad;
       t += (int64_t)gridDim.x * blockDim.x)
    p.ld[(t / pad) * p.s_pad + p.S + (t % pad)] = make_float2(0.f, 0.f);
}

// ---------------------------------------------------------------------------
// softmax-side work of one warp on 32 columns of a sub-tile buffer
// ---------------------------------------------------------------------------

// dQ side: this thread's query row against 32 keys (key indices base..base+31).
// Keeps key x iff x < A1 or B0 <= x < B1 (indices relative to base); writes
// dS = P (dP - D) as bf16 pairs over the first 16 of the 32 dP columns.
template <bool MASK>
__device__ __forceinline__ void ds_row(uint32_t tS, uint32_t tP, float scale_log2, float lse2,
                                       float drow, int32_t A1, int32_t B0, int32_t B1) {
  uint32_t sv[32], pv[32];
  tc::ld32(tS, sv);
  tc::ld32(tP, pv);
  tc::wait_ld();
  uint32_t packed[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float x0, x1, t0, t1, d0, d1;
    ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), scale_log2, scale_log2,
          -lse2, -lse2);
    x0 = ex2(x0);
    x1 = ex2(x1);
    fadd2(t0, t1, __uint_as_float(pv[e]), __uint_as_float(pv[e + 1]), -drow, -drow);
    fmul2(d0, d1, x0, x1, t0, t1);
    if (MASK) {
      d0 = ((e < A1) || (e >= B0 && e < B1)) ? d0 : 0.f;
      d1 = ((e + 1 < A1) || (e + 1 >= B0 && e + 1 < B1)) ? d1 : 0.f;
    }
    packed[e / 2] = pack_bf16(d0, d1);
  }
  tc::st16(tP, packed);
}

// dK/dV side: this thread's key row against 32 queries whose {LSE*log2e, D}
// pairs are ld[0..31].  Keeps query e iff LO <= e <= HI.  Writes P^T over the
// S^T columns and dS^T over the dP^T columns, as bf16 pairs.
template <bool MASK>
__device__ __forceinline__ void ds_col(uint32_t tS, uint32_t tP, float scale_log2,
                                       const float4* ld, int32_t LO, int32_t HI) {
  uint32_t sv[32], pv[32];
  tc::ld32(tS, sv);
  tc::ld32(tP, pv);
  tc::wait_ld();
  uint32_t pk_p[16], pk_s[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float4 l = ld[e / 2];  // {lse2_e, D_e, lse2_e+1, D_e+1}, same address on every lane
    float x0, x1, t0, t1, d0, d1;
    ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), scale_log2, scale_log2,
          -l.x, -l.z);
    x0 = ex2(x0);
    x1 = ex2(x1);
    fadd2(t0, t1, __uint_as_float(pv[e]), __uint_as_float(pv[e + 1]), -l.y, -l.w);
    if (MASK) {
      x0 = (e >= LO && e <= HI) ? x0 : 0.f;
      x1 = (e + 1 >= LO && e + 1 <= HI) ? x1 : 0.f;
    }
    fmul2(d0, d1, x0, x1, t0, t1);
    pk_p[e / 2] = pack_bf16(x0, x1);
    pk_s[e / 2] = pack_bf16(d0, d1);
  }
  tc::st16(tS, pk_p);
  tc::st16(tP, pk_s);
}

// ---------------------------------------------------------------------------
// 2a. dK/dV CTA: key tile kt of KV head hk, batch row b
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dkdv_cta(const Params& p, uint8_t* smem, Bars* bar, uint32_t tmem,
                                         int u) {
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTileR;
  uint8_t* sQ = smem + 2 * kTileR;  // stage st: Q at sQ + st * kStage, dO kTileC after it
  float2* sLd = reinterpret_cast<float2*>(smem + 2 * kTileR + kSt * kStage);  // [kSt][kBC]
  volatile int32_t* abort = &bar->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int per = p.hkv * p.B;
  const int kt = u / per;  // prefix tiles (the longest) first
  const int hk = (u % per) % p.hkv, b = (u % per) / p.hkv;
  const int G = p.hq / p.hkv;
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, false);
  const int32_t k0r = kt * kBM, k1r = min(p.S, k0r + kBM) - 1;
  // query sub-tiles that can admit one of these keys: from the one holding the
  // first key on; prefix keys are seen by every later query, window keys only
  // by queries at most W - 1 rows later
  const int n_qs = (p.S + kBC - 1) / kBC;
  const int qs_begin = k0r / kBC;
  int qs_end = n_qs;
  if ((int64_t)c0 + k0r >= P) qs_end = (int)min((int64_t)n_qs, ((int64_t)k1r + p.W - 1) / kBC + 1);
  const int n = max(0, qs_end - qs_begin) * G;  // (query sub-tile, head of the group) pairs

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&p.tmk_r);
      prefetch_tmap(&p.tmv_r);
      prefetch_tmap(&p.tmq_c);
      prefetch_tmap(&p.tmdo_c);
      const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
      mbar_arrive_expect_tx(&bar->res_full, 2 * kTileR);
      tma_load_4d(sK, &p.tmk_r, &bar->res_full, 0, hk, k0r, b, pol_kv);
      tma_load_4d(sK + kHalfR, &p.tmk_r, &bar->res_full, 64, hk, k0r, b, pol_kv);
      tma_load_4d(sV, &p.tmv_r, &bar->res_full, 0, hk, k0r, b, pol_kv);
      tma_load_4d(sV + kHalfR, &p.tmv_r, &bar->res_full, 64, hk, k0r, b, pol_kv);
      for (int i = 0; i < n; ++i) {
        const int st = i % kSt;
        if (!mbar_wait_abort(&bar->st_empty[st], ((i / kSt) & 1) ^ 1, abort)) break;
        const int qs = qs_begin + i / G, h = hk * G + i % G;
        uint8_t* dq = sQ + st * kStage;
        uint64_t* full = &bar->st_full[st];
        mbar_arrive_expect_tx(full, kStage + kLdBytes);
        tma_load_4d(dq, &p.tmq_c, full, 0, h, qs * kBC, b, pol_q);
        tma_load_4d(dq + kHalfC, &p.tmq_c, full, 64, h, qs * kBC, b, pol_q);
        tma_load_4d(dq + kTileC, &p.tmdo_c, full, 0, h, qs * kBC, b, pol_q);
        tma_load_4d(dq + kTileC + kHalfC, &p.tmdo_c, full, 64, h, qs * kBC, b, pol_q);
        bulk_load(sLd + st * kBC, p.ld + ((int64_t)b * p.hq + h) * p.s_pad + qs * kBC, kLdBytes,
                  full);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint64_t aK = tc::sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t aV = tc::sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t bQ = tc::sdesc_sw128(smem_u32(sQ), 16, 1024);            // K-major B
      const uint64_t bO = tc::sdesc_sw128(smem_u32(sQ + kTileC), 16, 1024);
      const uint64_t bQm = tc::sdesc_sw128(smem_u32(sQ), kHalfC, 1024);       // MN-major B
      const uint64_t bOm = tc::sdesc_sw128(smem_u32(sQ + kTileC), kHalfC, 1024);
      // S^T = K Q^T and dP^T = V dO^T of sub-tile i into buffer i & 1
      auto sdp = [&](int i) -> bool {
        const int st = i % kSt, bf = i & 1;
        if (!mbar_wait_abort(&bar->st_full[st], (i / kSt) & 1, abort)) return false;
        tc::fence_after();
        const uint64_t so = (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t oa = ((kk >> 2) * kHalfR + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * kHalfC + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tmem + bf * 128, aK + oa, bQ + so + ob, kIdescSub, kk > 0);
          tc::mma_bf16(tmem + bf * 128 + 64, aV + oa, bO + so + ob, kIdescSub, kk > 0);
        }
        tc::commit(smem_u32(&bar->s_full[bf]));
        return true;
      };
      // dV += P^T dO and dK += dS^T Q of sub-tile i, then release its stage
      auto acc = [&](int i) -> bool {
        const int st = i % kSt, bf = i & 1;
        if (!mbar_wait_abort(&bar->ds_ready[bf], (i >> 1) & 1, abort)) return false;
        tc::fence_after();
        const uint64_t so = (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBC / 16; ++kk) {
          const uint32_t ob = (kk * 2048) >> 4;
          tc::mma_bf16_ts(tmem + kTAcc, tmem + bf * 128 + packed_col(kk), bOm + so + ob,
                          kIdescAcc, i > 0 || kk > 0);
          tc::mma_bf16_ts(tmem + kTAcc + 128, tmem + bf * 128 + 64 + packed_col(kk),
                          bQm + so + ob, kIdescAcc, i > 0 || kk > 0);
        }
        tc::commit(smem_u32(&bar->st_empty[st]));
        return true;
      };
      bool ok = mbar_wait_abort(&bar->res_full, 0, abort);
      for (int i = 0; ok && i < n; ++i) {
        ok = sdp(i);
        if (ok && i > 0) ok = acc(i - 1);
      }
      if (ok) ok = acc(n - 1);
      if (ok) tc::commit(smem_u32(&bar->done));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t kpos = (int64_t)c0 + k0r + row;
    // queries that admit this key: positions [kpos, kend]
    const int64_t kend = kpos < P ? INT64_MAX / 2 : kpos + p.W - 1;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int st = i % kSt, bf = i & 1;
      const int qs = qs_begin + i / G;
      const int32_t qa = qs * kBC, qb = min(p.S, qa + kBC) - 1;
      const bool masked = qa + kBC > p.S ||
                          tile_class(km, c0, qa, qb, k0r, k1r, P, p.W) != kFull;
      // this warp's 32 queries: rows r0 + e, e = 0..31
      const int32_t r0 = qa + half * 32;
      const int64_t qp0 = (int64_t)c0 + r0;
      const int64_t lo64 = kpos - qp0;
      int64_t hi64 = kend - qp0;
      if (hi64 > (int64_t)(p.S - 1 - r0)) hi64 = (int64_t)(p.S - 1 - r0);
      const int32_t lo = (int32_t)(lo64 < 0 ? 0 : (lo64 > 32 ? 32 : lo64));
      const int32_t hi = (int32_t)(hi64 < -1 ? -1 : (hi64 > 31 ? 31 : hi64));
      ok = mbar_wait_abort(&bar->s_full[bf], (i >> 1) & 1, abort) &&
           mbar_wait_abort(&bar->st_full[st], (i / kSt) & 1, abort);  // the LSE / D pairs
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const float4* ld = reinterpret_cast<const float4*>(sLd + st * kBC + half * 32);
      const uint32_t tS = tmem + bf * 128 + half * 32 + lane_off;
      if (masked)
        ds_col<true>(tS, tS + 64, p.scale_log2, ld, lo, hi);
      else
        ds_col<false>(tS, tS + 64, p.scale_log2, ld, 0, 31);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->ds_ready[bf]);
    }
    if (ok && n > 0) {
      ok = mbar_wait_abort(&bar->done, 0, abort);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc::fence_after();
      const bool valid = k0r + row <= k1r;
      const int64_t base = (((int64_t)b * p.S + (valid ? k0r + row : 0)) * p.hkv + hk) * kHD;
      if (n > 0) {
        store_chunk(tmem + kTAcc + lane_off, p.dv + base, half, valid, 1.f, false, 0, p.turns);
        store_chunk(tmem + kTAcc + 128 + lane_off, p.dk + base, half, valid, p.scale, true,
                    (int32_t)kpos, p.turns);
      } else if (valid) {  // no query admits these keys: zero gradients
        for (int e = half * 32; e < half * 32 + 32; e += 4) {
          *reinterpret_cast<float4*>(p.dv + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dv + base + 64 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dk + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dk + base + 64 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2b. dQ CTA: query tile of head h, batch row b
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dq_cta(const Params& p, uint8_t* smem, Bars* bar, uint32_t tmem,
                                       int u) {
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + kTileR;
  uint8_t* sK = smem + 2 * kTileR;  // stage st: K at sK + st * kStage, V kTileC after it
  volatile int32_t* abort = &bar->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int per = p.hq * p.B;
  const int qt = p.nq - 1 - u / per;  // longest rows first
  const int h = (u % per) % p.hq, b = (u % per) / p.hq;
  const int hk = h / (p.hq / p.hkv);
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, false);
  const int32_t q0r = qt * kBM, q1r = min(p.S, q0r + kBM) - 1;
  const int64_t q0 = (int64_t)c0 + q0r, q1 = (int64_t)c0 + q1r;
  // 64-key sub-tiles that can hold an admitted pair: prefix ones, then the band
  const int32_t kc = keys_below(km, q1 + 1);
  const int32_t kP = keys_below(km, P);
  const int t1_end = (min(kP, kc) + kBC - 1) / kBC;
  const int32_t kw = keys_below(km, q0 - p.W + 1);
  const int t2_begin = max(t1_end, kw / kBC);
  const int t2_end = (kc + kBC - 1) / kBC;
  const int n = t1_end + max(0, t2_end - t2_begin);
  auto sub_at = [&](int i) { return i < t1_end ? i : t2_begin + (i - t1_end); };

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&p.tmq_r);
      prefetch_tmap(&p.tmdo_r);
      prefetch_tmap(&p.tmk_c);
      prefetch_tmap(&p.tmv_c);
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(&bar->res_full, 2 * kTileR);
      tma_load_4d(sQ, &p.tmq_r, &bar->res_full, 0, h, q0r, b, pol_q);
      tma_load_4d(sQ + kHalfR, &p.tmq_r, &bar->res_full, 64, h, q0r, b, pol_q);
      tma_load_4d(sdO, &p.tmdo_r, &bar->res_full, 0, h, q0r, b, pol_q);
      tma_load_4d(sdO + kHalfR, &p.tmdo_r, &bar->res_full, 64, h, q0r, b, pol_q);
      for (int i = 0; i < n; ++i) {
        const int st = i % kSt;
        if (!mbar_wait_abort(&bar->st_empty[st], ((i / kSt) & 1) ^ 1, abort)) break;
        const int ka = sub_at(i) * kBC;
        uint8_t* dk = sK + st * kStage;
        uint64_t* full = &bar->st_full[st];
        mbar_arrive_expect_tx(full, kStage);
        tma_load_4d(dk, &p.tmk_c, full, 0, hk, ka, b, pol_kv);
        tma_load_4d(dk + kHalfC, &p.tmk_c, full, 64, hk, ka, b, pol_kv);
        tma_load_4d(dk + kTileC, &p.tmv_c, full, 0, hk, ka, b, pol_kv);
        tma_load_4d(dk + kTileC + kHalfC, &p.tmv_c, full, 64, hk, ka, b, pol_kv);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint64_t aQ = tc::sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t aO = tc::sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t bK = tc::sdesc_sw128(smem_u32(sK), 16, 1024);               // K-major B
      const uint64_t bV = tc::sdesc_sw128(smem_u32(sK + kTileC), 16, 1024);
      const uint64_t bKm = tc::sdesc_sw128(smem_u32(sK), kHalfC, 1024);          // MN-major B
      // S = Q K^T and dP = dO V^T of sub-tile i into buffer i & 1
      auto sdp = [&](int i) -> bool {
        const int st = i % kSt, bf = i & 1;
        if (!mbar_wait_abort(&bar->st_full[st], (i / kSt) & 1, abort)) return false;
        tc::fence_after();
        const uint64_t so = (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t oa = ((kk >> 2) * kHalfR + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * kHalfC + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tmem + bf * 128, aQ + oa, bK + so + ob, kIdescSub, kk > 0);
          tc::mma_bf16(tmem + bf * 128 + 64, aO + oa, bV + so + ob, kIdescSub, kk > 0);
        }
        tc::commit(smem_u32(&bar->s_full[bf]));
        return true;
      };
      // dQ += dS K of sub-tile i, then release its stage
      auto acc = [&](int i) -> bool {
        const int st = i % kSt, bf = i & 1;
        if (!mbar_wait_abort(&bar->ds_ready[bf], (i >> 1) & 1, abort)) return false;
        tc::fence_after();
        const uint64_t so = (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBC / 16; ++kk)
          tc::mma_bf16_ts(tmem + kTAcc, tmem + bf * 128 + 64 + packed_col(kk),
                          bKm + so + ((kk * 2048) >> 4), kIdescAcc, i > 0 || kk > 0);
        tc::commit(smem_u32(&bar->st_empty[st]));
        return true;
      };
      bool ok = mbar_wait_abort(&bar->res_full, 0, abort);
      for (int i = 0; ok && i < n; ++i) {
        ok = sdp(i);
        if (ok && i > 0) ok = acc(i - 1);
      }
      if (ok) ok = acc(n - 1);
      if (ok) tc::commit(smem_u32(&bar->done));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t qpos = q0 + row;
    const float2 ldr = p.ld[((int64_t)b * p.hq + h) * p.s_pad + q0r + row];  // rows < s_pad
    // admitted key indices of this row: [0, a1) and [b0, b1)
    const int32_t a1 = keys_below(km, min((int64_t)P, qpos + 1));
    const int32_t b0 = keys_below(km, max((int64_t)0, qpos - p.W + 1));
    const int32_t b1 = keys_below(km, qpos + 1);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int bf = i & 1;
      const int32_t ka = sub_at(i) * kBC;
      const int32_t kb = min(km.n_keys, ka + kBC) - 1;
      const bool masked = ka + kBC > km.n_keys ||
                          tile_class(km, c0, q0r, q1r, ka, kb, P, p.W) != kFull;
      const int32_t base = ka + half * 32;
      ok = mbar_wait_abort(&bar->s_full[bf], (i >> 1) & 1, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const uint32_t tS = tmem + bf * 128 + half * 32 + lane_off;
      if (masked)
        ds_row<true>(tS, tS + 64, p.scale_log2, ldr.x, ldr.y, a1 - base, b0 - base, b1 - base);
      else
        ds_row<false>(tS, tS + 64, p.scale_log2, ldr.x, ldr.y, 0, 0, 0);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->ds_ready[bf]);
    }
    if (ok && n > 0) {
      ok = mbar_wait_abort(&bar->done, 0, abort);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc::fence_after();
      const bool valid = q0r + row <= q1r;
      float* dst = p.dq + (((int64_t)b * p.S + (valid ? q0r + row : 0)) * p.hq + h) * kHD;
      if (n > 0) {
        store_chunk(tmem + kTAcc + lane_off, dst, half, valid, p.scale, true, (int32_t)qpos,
                    p.turns);
      } else if (valid) {
        for (int e = half * 32; e < half * 32 + 32; e += 4) {
          *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dst + 64 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) bwd_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  Bars* bar = reinterpret_cast<Bars*>(smem + 2 * kTileR + kSt * kStage + kSt * kLdBytes);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::alloc(smem_u32(&bar->tmem_slot), 512);
    tc::relinquish();
  }
  if (tid == 32) {
    mbar_init(&bar->res_full, 1);
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&bar->st_full[s], 1);
      mbar_init(&bar->st_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->ds_ready[i], 8);  // one arrival per softmax warp
    }
    mbar_init(&bar->done, 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bar->tmem_slot;
  grid_dependency_wait();  // rotated Q / K and the LSE / D pairs come from the pre-pass

  const int u = (int)blockIdx.x;
  if (u < p.n_dkdv)
    dkdv_cta(p, smem, bar, tmem, u);
  else
    dq_cta(p, smem, bar, tmem, u - p.n_dkdv);

  tc::fence_before();
  __syncthreads();
  if (bar->abort) {
    if (tid == 0) set_flag(p.status, PS_DEV_TIMEOUT);
    // copies and products already issued finish on their own within microseconds;
    // give them time before the CTA's shared and tensor memory are released
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
  size_t q_off, k_off, ld_off, total;
  int32_t s_pad;
};

static Layout layout(int B, int S, int hq, int hkv, int D) {
  Layout L;
  L.s_pad = (S + kBM - 1) / kBM * kBM;
  L.q_off = 0;
  L.k_off = align256((size_t)B * S * hq * D * 2);
  L.ld_off = L.k_off + align256((size_t)B * S * hkv * D * 2);
  L.total = L.ld_off + align256((size_t)B * hq * L.s_pad * 8);
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
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(d_out) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return PS_ERR_ALIGNMENT;
  const bwd::Layout L = bwd::layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PS_ERR_WORKSPACE;
  if (workspace_bytes < L.total) return PS_ERR_WORKSPACE;
  const int32_t nq = (seqlen + bwd::kBM - 1) / bwd::kBM;
  const int64_t n_dkdv = (int64_t)nq * n_kv_heads * batch;
  const int64_t n_dq = (int64_t)nq * n_q_heads * batch;
  if (n_dkdv + n_dq > 0x7fffffffLL) return PS_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;

  bwd::PrepParams g;
  g.q = static_cast<const uint4*>(q);
  g.k = static_cast<const uint4*>(k);
  g.o = static_cast<const uint4*>(out);
  g.dout = static_cast<const uint4*>(d_out);
  g.lse = lse;
  g.qh = reinterpret_cast<uint4*>(ws + L.q_off);
  g.kh = reinterpret_cast<uint4*>(ws + L.k_off);
  g.ld = reinterpret_cast<float2*>(ws + L.ld_off);
  g.q_start = q_start;
  g.B = batch;
  g.S = seqlen;
  g.s_pad = L.s_pad;
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
  const uint32_t box_r[4] = {64u, 1u, (uint32_t)bwd::kBM, 1u};
  const uint32_t box_c[4] = {64u, 1u, (uint32_t)bwd::kBC, 1u};
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool okm = encode_tmap(&p.tmq_r, bf, 4, ws + L.q_off, qd, qs, box_r, sw) &&
                   encode_tmap(&p.tmq_c, bf, 4, ws + L.q_off, qd, qs, box_c, sw) &&
                   encode_tmap(&p.tmdo_r, bf, 4, d_out, qd, qs, box_r, sw) &&
                   encode_tmap(&p.tmdo_c, bf, 4, d_out, qd, qs, box_c, sw) &&
                   encode_tmap(&p.tmk_r, bf, 4, ws + L.k_off, kd, ks, box_r, sw) &&
                   encode_tmap(&p.tmk_c, bf, 4, ws + L.k_off, kd, ks, box_c, sw) &&
                   encode_tmap(&p.tmv_r, bf, 4, v, kd, ks, box_r, sw) &&
                   encode_tmap(&p.tmv_c, bf, 4, v, kd, ks, box_c, sw);
  if (!okm) return PS_ERR_CUDA;
  p.ld = reinterpret_cast<const float2*>(ws + L.ld_off);
  p.q_start = q_start;
  p.prefix_len = prefix_len;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.S = seqlen;
  p.s_pad = L.s_pad;
  p.hq = n_q_heads;
  p.hkv = n_kv_heads;
  p.W = window;
  p.B = batch;
  p.nq = nq;
  p.n_dkdv = (int32_t)n_dkdv;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  make_rope_turns(rope_theta, head_dim, &p.turns);
  if (cudaFuncSetAttribute(bwd::bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bwd::kSmem) != cudaSuccess)
    return PS_ERR_CUDA;
  if (launch_dependent(bwd::bwd_kernel, dim3((unsigned)(n_dkdv + n_dq)), dim3(bwd::kThreads),
                       (size_t)bwd::kSmem, s, p) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}
