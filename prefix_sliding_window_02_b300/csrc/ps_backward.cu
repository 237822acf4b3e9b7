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
//         K and V stay in shared memory while 128-query tiles of Q and dO of
//         every query head of the group stream past;
//       dQ CTAs, one per (128-query tile, query head, batch row): Q and dO stay
//         while the forward's 128-key tiles of K and V stream past.
//     Both recompute S and dP, so each (query, key) tile pair costs 7 products
//     instead of the 5 of a single pass that adds dQ with atomics.
//
// Every product is a tcgen05 MMA with M = N = 128: on this tensor core one
// instruction costs about the same pipe time for N = 64 as for N = 128, so
// narrower products would halve the rate.  TMEM (512 columns) holds two step
// buffers of 128 columns and the fp32 accumulators (dV | dK, or dQ).  A step
// (one streamed tile) runs in its buffer: S is computed there, the softmax
// warps turn it into P (kept in registers), dP then overwrites the buffer, and
// the softmax warps turn it into dS, written back as bf16 pairs over the first
// half of each warp's columns, the tensor-memory A operand of dQ += dS K or
// dK += dS^T Q.  In a dK/dV CTA P^T also goes back as bf16 for dV += P^T dO,
// into the other buffer's second halves (columns of the previous step's dP^T
// already consumed), so that dP^T(t) need not wait for dV(t).  The issuer
// orders the products dP(t), S(t+1), dQ(t) in a dQ CTA and dP^T(t), dV(t),
// S^T(t+1), dK(t) in a dK/dV CTA: S(t+1) runs while the softmax warps compute
// dS(t), and dS(t)'s product while they compute P(t+1).  Tensor-core
// instructions of one thread execute in issue order, which lets a product
// overwrite a buffer that an earlier product has just read.
//
// CTA roles (320 threads): warps 0-7 are the softmax warps (two per TMEM lane
// quadrant, each on 64 of a step's 128 columns), warp 8 issues the TMA copies,
// warp 9 issues the MMAs.
#include "ps_internal.h"
#include "ps_math.cuh"
#include "ps_rope.cuh"
#include "ps_tc.cuh"
#include "ps_tiles.cuh"

namespace ps {
namespace bwd {

constexpr int kT = 128;                  // rows of every tile (resident and streamed)
constexpr int kHalf = kT * 128;          // one 64-column swizzled half of a tile: 16 KB
constexpr int kTile = 2 * kHalf;         // one slot: 32 KB, sized for head dim 128
constexpr int kLdBytes = kT * 8;         // {LSE*log2e, D} pairs of one query tile
constexpr int kSoftWarps = 8;
constexpr int kParts = kSoftWarps / 4;   // softmax warps per TMEM lane quadrant
constexpr int kNC = kT / kParts;         // step columns per softmax warp
constexpr int kProducerWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;
constexpr int kThreads = 32 * (kSoftWarps + 2);
// Streamed tiles: ring A holds the operand used by S(t) and by the last
// product of step t (K in a dQ CTA, Q in a dK/dV CTA), ring B the one used by
// dP(t) (V, or dO).  A slot of ring A frees late, so a dQ CTA gives it three
// slots; a dK/dV CTA also stages the query tile's LSE / D pairs and has room
// for two.
constexpr int kSaQ = 3, kSaKV = 2, kSb = 2;
constexpr int kOffA = 2 * kTile;                 // ring A, after the two resident tiles
constexpr int kOffB = kOffA + kSaQ * kTile;      // ring B (same place in both roles)
constexpr int kOffLd = kOffA + kSaKV * kTile;    // dK/dV: LSE / D slots, where a dQ CTA
                                                 // has its third ring-A slot
constexpr int kOffBars = kOffB + kSb * kTile;
constexpr int kSmem = kOffBars + 256 /*barriers*/ + 1024 /*alignment*/;
static_assert(kOffLd + kSaKV * kLdBytes <= kOffB, "LSE / D slots fit in the spare slot");
constexpr uint32_t kIdescS = tc::idesc_bf16(128, 128, false);   // S, dP: both operands K-major
constexpr uint32_t kTAcc = 256;                                  // accumulator columns
// dK/dV CTA: P^T(t) is packed into the second half of each softmax warp's column
// share of the other step buffer (the first half of each share holds dS^T)
constexpr uint32_t kPOff = kNC / 2;

// Per head dim D (64 or 128): the bytes a 128-row tile fills of its slot, its
// 64-column halves, the accumulations' instruction descriptor (N = D, B
// MN-major) and the rotation pairs each softmax warp writes in the epilogue.
template <int D>
struct Geo {
  static constexpr int kBytes = kT * D * 2;
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kIdescAcc = tc::idesc_bf16(128, D, true);
  static constexpr int kPairs = D / 2 / kParts;
};

struct Params {
  CUtensorMap tmq, tmdo;  // rotated Q, dO  {D, Hq, S, B}, 128-row boxes
  CUtensorMap tmk, tmv;   // rotated K, V   {D, Hkv, S, B}
  // head dim 128: fp32 gradients {D, H, S, B}, 32 x 32 boxes, 128-byte swizzle
  CUtensorMap tmdq, tmdk, tmdv;
  const float2* ld;       // [B, Hq, s_pad] {LSE * log2(e), D}; rows >= S are zero
  const int32_t* q_start;
  const int32_t* prefix_len;
  float* dq;  // [B, S, Hq, D]
  float* dk;  // [B, S, Hkv, D]
  float* dv;  // [B, S, Hkv, D]
  int32_t* status;
  int32_t S, s_pad, hq, hkv, W, B;
  int32_t nq;       // 128-row tiles
  int32_t n_dkdv;   // CTAs of the dK/dV kind (the first ones of the grid)
  float scale, scale_log2;
  uint64_t wait_ns;          // bounded-wait limit
  int32_t drop_first_load;   // test hook: CTA 0 skips its first streamed copy
  RopeTurns turns;
};

struct Bars {
  uint64_t res_full;                         // the resident tiles have landed
  uint64_t a_full[kSaQ], a_empty[kSaQ];      // ring A
  uint64_t b_full[kSb], b_empty[kSb];        // ring B
  uint64_t s_full[2], p_ready[2];            // step buffers: S computed / P taken
  uint64_t dp_full[2], ds_ready[2];          //               dP computed / dS written
  uint64_t done;                             // every product has completed
  uint64_t drain;                            // after an abort: the issuer's products completed
  uint32_t tmem_slot;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// The copies the producer has issued, for the drain after an abort: whether the
// resident tiles were requested, and the phase parity of the last load into
// each slot of rings A and B (-1: none).
struct Inflight {
  int res;
  int a[kSaQ];
  int b[kSb];
};

__device__ __forceinline__ void tld(uint32_t taddr, uint32_t (&r)[32]) { tc::ld32(taddr, r); }
__device__ __forceinline__ void tld(uint32_t taddr, uint32_t (&r)[16]) { tc::ld16(taddr, r); }

// TMEM column of the K16 step kk (16 step columns) of the bf16 pairs the
// softmax warps write over a buffer: the warp on columns [c0, c0 + kNC) packs
// them into [c0, c0 + kNC / 2).
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return (16 * kk) / kNC * kNC + (16 * kk) % kNC / 2;
}

// Writes NP rotation pairs (chunk c: columns [c NP, (c+1) NP) with their
// partners D/2 further on) of one thread's row of a D-wide fp32 accumulator,
// scaled and rotated back by -pos when `rot` (dQ, dK), plainly otherwise (dV).
// Every thread of the warp calls it (tcgen05.ld is warp-collective); only rows
// with `valid` store.
template <int D>
__device__ __forceinline__ void store_chunk(uint32_t taddr, float* dst, int c, bool valid, float mul,
                                            bool rot, int32_t pos, const RopeTurns& turns) {
  constexpr int kPairs = Geo<D>::kPairs, kH = D / 2;
  uint32_t a[kPairs], b[kPairs];
  tld(taddr + c * kPairs, a);
  tld(taddr + kH + c * kPairs, b);
  tc::wait_ld();
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < kPairs; ++e) {
    const float x = __uint_as_float(a[e]) * mul, y = __uint_as_float(b[e]) * mul;
    float rx = x, ry = y;
    if (rot) {
      float cs, sn;
      rope_cos_sin(pos, turns.f[c * kPairs + e], cs, sn);
      rx = x * cs + y * sn;  // rotation by -angle
      ry = y * cs - x * sn;
    }
    a[e] = __float_as_uint(rx);
    b[e] = __float_as_uint(ry);
  }
#pragma unroll
  for (int e = 0; e < kPairs; e += 4) {
    *reinterpret_cast<uint4*>(dst + c * kPairs + e) = make_uint4(a[e], a[e + 1], a[e + 2], a[e + 3]);
    *reinterpret_cast<uint4*>(dst + kH + c * kPairs + e) =
        make_uint4(b[e], b[e + 1], b[e + 2], b[e + 3]);
  }
}

// Head dim 128: the same values as store_chunk for the warp's 32 rows (lanes),
// written through shared memory and two tensor stores (columns [32 c, 32 c + 32)
// and their partners 64 further on), so that each store moves whole 128-byte
// row segments instead of one 16-byte piece per row.  `stage` (8 KB,
// 1024-byte aligned) holds the two 32 x 32 fp32 boxes in the 128-byte swizzled
// layout of the tensor map.  Rows past the tensor's end are clipped by the
// store.  Lane 0 commits the stores; the caller waits for them to have read
// shared memory before it is reused or released.
__device__ __forceinline__ void store_chunk_tma(uint32_t taddr, uint8_t* stage,
                                                const CUtensorMap* map, int c, float mul, bool rot,
                                                int32_t pos, const RopeTurns& turns, int32_t head,
                                                int32_t row0, int32_t b, int lane) {
  constexpr int kPairs = 32, kH = 64;
  uint32_t a[kPairs], v[kPairs];
  tld(taddr + c * kPairs, a);
  tld(taddr + kH + c * kPairs, v);
  tc::wait_ld();
#pragma unroll
  for (int e = 0; e < kPairs; ++e) {
    const float x = __uint_as_float(a[e]) * mul, y = __uint_as_float(v[e]) * mul;
    float rx = x, ry = y;
    if (rot) {
      float cs, sn;
      rope_cos_sin(pos, turns.f[c * kPairs + e], cs, sn);
      rx = x * cs + y * sn;  // rotation by -angle
      ry = y * cs - x * sn;
    }
    a[e] = __float_as_uint(rx);
    v[e] = __float_as_uint(ry);
  }
  const uint32_t s0 = smem_u32(stage);
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of this row, swizzled
    const uint32_t off = lane * 128 + ((j ^ (lane & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(s0 + off), "r"(a[4 * j]),
                 "r"(a[4 * j + 1]), "r"(a[4 * j + 2]), "r"(a[4 * j + 3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(s0 + 4096 + off),
                 "r"(v[4 * j]), "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                 : "memory");
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_4d(map, stage, c * kPairs, head, row0, b);
    tma_store_4d(map, stage + 4096, kH + c * kPairs, head, row0, b);
    bulk_commit();
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
  int32_t rotate;  // 0: the forward's rotated Q and K are reused, only D is computed
  RopeTurns turns;
};

constexpr int kPrepRows = 16;

// One block takes kPrepRows rows (batch row, position) at a time: the angles
// of those rows, then every 16-byte group of their Q and K rows, then D for
// every (row, query head) with a half-warp per pair (8 elements per lane).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  constexpr int VEC = D / 8, HALFV = D / 16, NPAIR = D / 2, NG = D / 16;
  __shared__ float2 cs[kPrepRows][NPAIR];
  grid_dependency_wait();
  allow_dependents();
  const int64_t n_rows = (int64_t)p.B * p.S;
  const int heads = p.rotate ? p.hq + p.hkv : 0;
  for (int64_t r0 = (int64_t)blockIdx.x * kPrepRows; r0 < n_rows;
       r0 += (int64_t)gridDim.x * kPrepRows) {
    for (int t = threadIdx.x; t < (p.rotate ? kPrepRows * NPAIR : 0); t += blockDim.x) {
      const int rr = t / NPAIR, i = t % NPAIR;
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
    for (int it = threadIdx.x; it < kPrepRows * heads * NG; it += blockDim.x) {
      const int g = it % NG;
      const int hd = (it / NG) % heads;
      const int rr = (it / NG) / heads;
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
    // D_i = dO_i . O_i and the stored pair, one half-warp per (row, query head)
    const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    for (int w = hw; w < kPrepRows * p.hq; w += blockDim.x / 16) {
      const int64_t r = r0 + w / p.hq;
      const int h = w % p.hq;
      float acc = 0.f;
      if (r < n_rows && l16 < VEC) {  // 8 elements per lane
        const uint4 a = p.o[(r * p.hq + h) * VEC + l16], d = p.dout[(r * p.hq + h) * VEC + l16];
        acc = bf16lo(a.x) * bf16lo(d.x) + bf16hi(a.x) * bf16hi(d.x) + bf16lo(a.y) * bf16lo(d.y) +
              bf16hi(a.y) * bf16hi(d.y) + bf16lo(a.z) * bf16lo(d.z) + bf16hi(a.z) * bf16hi(d.z) +
              bf16lo(a.w) * bf16lo(d.w) + bf16hi(a.w) * bf16hi(d.w);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (l16 == 0 && r < n_rows) {
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
// softmax-side work of one warp on its kNC columns of a step buffer
// ---------------------------------------------------------------------------

// dQ side, first half: this thread's query row against kNC keys (key indices
// base..).  P = exp2(S * scale_log2 - lse2), zero unless bit x of km is set
// (key x, relative to base, admitted); kept in registers.
template <bool MASK>
__device__ __forceinline__ void p_row(uint32_t tS, float scale_log2, float lse2,
                                      const uint32_t (&km)[kNC / 32], float (&pr)[kNC]) {
#pragma unroll
  for (int c = 0; c < kNC / 32; ++c) {
    uint32_t sv[32];
    tc::ld32(tS + 32 * c, sv);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int x = 32 * c + e;
      float x0, x1;
      ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), scale_log2, scale_log2,
            -lse2, -lse2);
      x0 = ex2(x0);
      x1 = ex2(x1);
      if (MASK) {
        x0 = (km[x >> 5] & (1u << (x & 31))) ? x0 : 0.f;
        x1 = (km[(x + 1) >> 5] & (1u << ((x + 1) & 31))) ? x1 : 0.f;
      }
      pr[x] = x0;
      pr[x + 1] = x1;
    }
  }
}

// dQ side, second half: dS = P (dP - D) over the same columns, written as
// bf16 pairs over the first kNC / 2 of them (32 columns at a time, each chunk
// packed into 16 columns the warp has already read).
__device__ __forceinline__ void ds_row(uint32_t tP, float drow, const float (&pr)[kNC]) {
#pragma unroll
  for (int c = 0; c < kNC / 32; ++c) {
    uint32_t pv[32];  // the bf16 pairs are packed into its first half as it is consumed
    tc::ld32(tP + 32 * c, pv);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float t0, t1, d0, d1;
      fadd2(t0, t1, __uint_as_float(pv[e]), __uint_as_float(pv[e + 1]), -drow, -drow);
      fmul2(d0, d1, pr[32 * c + e], pr[32 * c + e + 1], t0, t1);
      pv[e / 2] = pack_bf16(d0, d1);
    }
    tc::st16(tP + 16 * c, reinterpret_cast<const uint32_t(&)[16]>(pv));
  }
}

// dK/dV side, first half: this thread's key row against kNC queries whose
// {LSE*log2e, D} pairs are ld[0..kNC) (as float4: two queries each).  P^T is
// zero unless bit e of km is set (query e admits the key); kept in registers
// and written as kNC / 2 columns of bf16 pairs at tP for dV += P^T dO.
template <bool MASK>
__device__ __forceinline__ void p_col(uint32_t tS, uint32_t tP, float scale_log2,
                                      const float4* ld, const uint32_t (&km)[kNC / 32],
                                      float (&pr)[kNC]) {
#pragma unroll
  for (int c = 0; c < kNC / 32; ++c) {
    uint32_t sv[32];  // the bf16 pairs are packed into its first half as it is consumed
    tc::ld32(tS + 32 * c, sv);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int x = 32 * c + e;
      const float4 l = ld[x / 2];  // same address on every lane
      float x0, x1;
      ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), scale_log2, scale_log2,
            -l.x, -l.z);
      x0 = ex2(x0);
      x1 = ex2(x1);
      if (MASK) {
        x0 = (km[x >> 5] & (1u << (x & 31))) ? x0 : 0.f;
        x1 = (km[(x + 1) >> 5] & (1u << ((x + 1) & 31))) ? x1 : 0.f;
      }
      pr[x] = x0;
      pr[x + 1] = x1;
      sv[e / 2] = pack_bf16(x0, x1);
    }
    tc::st16(tP + 16 * c, reinterpret_cast<const uint32_t(&)[16]>(sv));
  }
}

// dK/dV side, second half: dS^T = P^T (dP^T - D) as bf16 pairs.
__device__ __forceinline__ void ds_col(uint32_t tP, const float4* ld, const float (&pr)[kNC]) {
#pragma unroll
  for (int c = 0; c < kNC / 32; ++c) {
    uint32_t pv[32];
    tc::ld32(tP + 32 * c, pv);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int x = 32 * c + e;
      const float4 l = ld[x / 2];
      float t0, t1, d0, d1;
      fadd2(t0, t1, __uint_as_float(pv[e]), __uint_as_float(pv[e + 1]), -l.y, -l.w);
      fmul2(d0, d1, pr[x], pr[x + 1], t0, t1);
      pv[e / 2] = pack_bf16(d0, d1);
    }
    tc::st16(tP + 16 * c, reinterpret_cast<const uint32_t(&)[16]>(pv));
  }
}

// Hands a step buffer from the softmax warps back to the issuer.
__device__ __forceinline__ void release(uint64_t* bar, int lane, bool stored) {
  if (stored) tc::wait_st();
  tc::fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// One 128 x 128 product over the head dim: D / 16 MMAs (K16 steps) into the
// accumulator d_tmem.
template <int D>
__device__ __forceinline__ void mma_ss8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        bool acc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
    tc::mma_bf16(d_tmem, adesc + off, bdesc + off, kIdescS, acc || kk > 0);
  }
}

// d_tmem (+)= A (bf16 pairs in TMEM at a_tmem, packed as the softmax warps
// write them) x B (128 rows of a tile, MN-major, N = D).
template <int D>
__device__ __forceinline__ void mma_ts8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc_mn,
                                        bool acc) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    tc::mma_bf16_ts(d_tmem, a_tmem + packed_col(kk), bdesc_mn + ((kk * 2048) >> 4),
                    Geo<D>::kIdescAcc, acc || kk > 0);
}

// ---------------------------------------------------------------------------
// 2a. dK/dV CTA: key tile kt of KV head hk, batch row b
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void dkdv_cta(const Params& p, uint8_t* smem, Bars* bar, uint32_t tmem,
                                         int u, Inflight& fl) {
  constexpr int kSa = kSaKV;
  constexpr int kB = Geo<D>::kBytes, kNH = Geo<D>::kHalves;
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sA = smem + kOffA;  // Q tiles
  uint8_t* sB = smem + kOffB;  // dO tiles
  float2* sLd = reinterpret_cast<float2*>(smem + kOffLd);  // [kSa][kT]
  volatile int32_t* abort = &bar->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int per = p.hkv * p.B;
  const int kt = u / per;  // prefix tiles (the longest) first
  const int hk = (u % per) % p.hkv, b = (u % per) / p.hkv;
  const int G = p.hq / p.hkv;
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, false);
  const int32_t k0r = kt * kT, k1r = min(p.S, k0r + kT) - 1;
  // query tiles that can admit one of these keys: from the tile holding the
  // first key on; prefix keys are seen by every later query, window keys only
  // by queries at most W - 1 rows later
  int qt_end = p.nq;
  if ((int64_t)c0 + k0r >= P) qt_end = (int)min((int64_t)p.nq, ((int64_t)k1r + p.W - 1) / kT + 1);
  const int n = max(0, qt_end - kt) * G;  // steps: (query tile, head of the group)

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&p.tmk);
      prefetch_tmap(&p.tmv);
      prefetch_tmap(&p.tmq);
      prefetch_tmap(&p.tmdo);
      const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
      mbar_arrive_expect_tx(&bar->res_full, 2 * kB);
      for (int x = 0; x < kNH; ++x) {
        tma_load_4d(sK + x * kHalf, &p.tmk, &bar->res_full, 64 * x, hk, k0r, b, pol_kv);
        tma_load_4d(sV + x * kHalf, &p.tmv, &bar->res_full, 64 * x, hk, k0r, b, pol_kv);
      }
      fl.res = 1;
      for (int t = 0; t < n; ++t) {
        const int qt = kt + t / G, h = hk * G + t % G;
        const int sa = t % kSa, sb = t % kSb;
        if (!mbar_wait_abort(&bar->a_empty[sa], ((t / kSa) & 1) ^ 1, abort, p.wait_ns)) break;
        uint64_t* fa = &bar->a_full[sa];
        // test hook: CTA 0 leaves its first ring-A slot without copy or arrival
        if (!(t == 0 && p.drop_first_load && blockIdx.x == 0)) {
          mbar_arrive_expect_tx(fa, kB + kLdBytes);
          for (int x = 0; x < kNH; ++x)
            tma_load_4d(sA + sa * kTile + x * kHalf, &p.tmq, fa, 64 * x, h, qt * kT, b, pol_q);
          bulk_load(sLd + sa * kT, p.ld + ((int64_t)b * p.hq + h) * p.s_pad + qt * kT, kLdBytes, fa);
          fl.a[sa] = (t / kSa) & 1;
        }
        if (!mbar_wait_abort(&bar->b_empty[sb], ((t / kSb) & 1) ^ 1, abort, p.wait_ns)) break;
        uint64_t* fb = &bar->b_full[sb];
        mbar_arrive_expect_tx(fb, kB);
        for (int x = 0; x < kNH; ++x)
          tma_load_4d(sB + sb * kTile + x * kHalf, &p.tmdo, fb, 64 * x, h, qt * kT, b, pol_q);
        fl.b[sb] = (t / kSb) & 1;
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint64_t aK = tc::sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t aV = tc::sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t bQ = tc::sdesc_sw128(smem_u32(sA), 16, 1024);       // K-major
      const uint64_t bQm = tc::sdesc_sw128(smem_u32(sA), kHalf, 1024);   // MN-major
      const uint64_t bO = tc::sdesc_sw128(smem_u32(sB), 16, 1024);
      const uint64_t bOm = tc::sdesc_sw128(smem_u32(sB), kHalf, 1024);
      auto soa = [](int t) { return (uint64_t)(((t % kSa) * kTile) >> 4); };
      auto sob = [](int t) { return (uint64_t)(((t % kSb) * kTile) >> 4); };
      // Per step t (buffer t & 1): dP^T = V dO^T, dV += P^T dO, S^T of step
      // t+1, then dK += dS^T Q.  The softmax warps write P^T(t) into the other
      // buffer's unused half -- the columns of dP^T(t-1) they have already
      // consumed, beside dS^T(t-1) -- so dP^T(t), on the path to dS^T(t), does
      // not wait for dV(t) to read P^T(t); S^T(t+1) then overwrites that buffer
      // after dV(t) and dK(t-1) have read it (one thread's products run in order).
      bool ok = mbar_wait_abort(&bar->res_full, 0, abort, p.wait_ns) &&
                mbar_wait_abort(&bar->a_full[0], 0, abort, p.wait_ns);
      if (ok) {
        tc::fence_after();
        mma_ss8<D>(tmem, aK, bQ + soa(0), false);  // S^T(0) = K Q(0)^T
        tc::commit(smem_u32(&bar->s_full[0]));
      }
      for (int t = 0; ok && t < n; ++t) {
        const int bf = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        const uint32_t tb = tmem + bf * 128;
        if (!(ok = mbar_wait_abort(&bar->p_ready[bf], ph, abort, p.wait_ns) &&
                   mbar_wait_abort(&bar->b_full[t % kSb], (t / kSb) & 1, abort, p.wait_ns)))
          break;
        tc::fence_after();
        mma_ss8<D>(tb, aV, bO + sob(t), false);  // dP^T = V dO^T
        tc::commit(smem_u32(&bar->dp_full[bf]));
        mma_ts8<D>(tmem + kTAcc, tmem + (bf ^ 1) * 128 + kPOff, bOm + sob(t), t > 0);  // dV
        tc::commit(smem_u32(&bar->b_empty[t % kSb]));
        if (t + 1 < n) {
          if (!(ok = mbar_wait_abort(&bar->a_full[(t + 1) % kSa], ((t + 1) / kSa) & 1, abort, p.wait_ns)))
            break;
          tc::fence_after();
          mma_ss8<D>(tmem + (bf ^ 1) * 128, aK, bQ + soa(t + 1), false);
          tc::commit(smem_u32(&bar->s_full[bf ^ 1]));
        }
        if (!(ok = mbar_wait_abort(&bar->ds_ready[bf], ph, abort, p.wait_ns))) break;
        tc::fence_after();
        mma_ts8<D>(tmem + kTAcc + 128, tb, bQm + soa(t), t > 0);  // dK += dS^T Q
        tc::commit(smem_u32(&bar->a_empty[t % kSa]));
      }
      if (ok) tc::commit(smem_u32(&bar->done));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, part = warp >> 2;
    const int row = quad * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t kpos = (int64_t)c0 + k0r + row;
    // queries that admit this key: positions [kpos, kend]
    const int64_t kend = kpos < P ? INT64_MAX / 2 : kpos + p.W - 1;
    bool ok = true;
    float pr[kNC];
    for (int t = 0; t < n; ++t) {
      const int bf = t & 1, sa = t % kSa;
      const uint32_t ph = (t >> 1) & 1;
      const int32_t qa = (kt + t / G) * kT, qb = min(p.S, qa + kT) - 1;
      const bool masked = qa + kT > p.S || tile_class(km, c0, qa, qb, k0r, k1r, P, p.W) != kFull;
      // this warp's kNC queries: rows r0 + e
      const int32_t r0 = qa + part * kNC;
      const int64_t qp0 = (int64_t)c0 + r0;
      const int64_t lo64 = kpos - qp0;
      int64_t hi64 = kend - qp0;
      if (hi64 > (int64_t)(p.S - 1 - r0)) hi64 = (int64_t)(p.S - 1 - r0);
      const int32_t lo = (int32_t)(lo64 < 0 ? 0 : (lo64 > kNC ? kNC : lo64));
      const int32_t hi = (int32_t)(hi64 < -1 ? -1 : (hi64 > kNC - 1 ? kNC - 1 : hi64));
      const uint32_t tS = tmem + bf * 128 + part * kNC + lane_off;
      const float4* ld = reinterpret_cast<const float4*>(sLd + sa * kT + part * kNC);
      uint32_t kmask[kNC / 32];
      if (masked) {
#pragma unroll
        for (int w = 0; w < kNC / 32; ++w) kmask[w] = keep_bits(32 * w, 0, lo, hi + 1);
      }
      ok = mbar_wait_abort(&bar->s_full[bf], ph, abort, p.wait_ns) &&
           mbar_wait_abort(&bar->a_full[sa], (t / kSa) & 1, abort, p.wait_ns);  // the LSE / D pairs
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      // P^T(t) goes to the other buffer, beside dS^T(t-1) (see the issuer)
      const uint32_t tPo = tmem + (bf ^ 1) * 128 + part * kNC + kPOff + lane_off;
      if (masked)
        p_col<true>(tS, tPo, p.scale_log2, ld, kmask, pr);
      else
        p_col<false>(tS, tPo, p.scale_log2, ld, kmask, pr);
      release(&bar->p_ready[bf], lane, true);
      ok = mbar_wait_abort(&bar->dp_full[bf], ph, abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      ds_col(tS, ld, pr);
      release(&bar->ds_ready[bf], lane, true);
    }
    if (ok && n > 0) {
      ok = mbar_wait_abort(&bar->done, 0, abort, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc::fence_after();
      const bool valid = k0r + row <= k1r;
      const int64_t base = (((int64_t)b * p.S + (valid ? k0r + row : 0)) * p.hkv + hk) * D;
      if (n > 0 && D == 128) {
        // staging in the operand rings, free now that every product has completed
        const int32_t row0 = k0r + quad * 32;
        store_chunk_tma(tmem + kTAcc + lane_off, smem + kOffA + warp * 8192, &p.tmdv, part, 1.f,
                        false, 0, p.turns, hk, row0, b, lane);
        store_chunk_tma(tmem + kTAcc + 128 + lane_off, smem + kOffB + warp * 8192, &p.tmdk, part,
                        p.scale, true, (int32_t)kpos, p.turns, hk, row0, b, lane);
        if (lane == 0) bulk_wait_read_all();
      } else if (n > 0) {
        store_chunk<D>(tmem + kTAcc + lane_off, p.dv + base, part, valid, 1.f, false, 0, p.turns);
        store_chunk<D>(tmem + kTAcc + 128 + lane_off, p.dk + base, part, valid, p.scale, true,
                       (int32_t)kpos, p.turns);
      } else if (valid) {  // no query admits these keys: zero gradients
        constexpr int kPairs = Geo<D>::kPairs;
        for (int e = part * kPairs; e < part * kPairs + kPairs; e += 4) {
          *reinterpret_cast<float4*>(p.dv + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dv + base + D / 2 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dk + base + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(p.dk + base + D / 2 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2b. dQ CTA: query tile of head h, batch row b
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void dq_cta(const Params& p, uint8_t* smem, Bars* bar, uint32_t tmem,
                                       int u, Inflight& fl) {
  constexpr int kSa = kSaQ;
  constexpr int kB = Geo<D>::kBytes, kNH = Geo<D>::kHalves;
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + kTile;
  uint8_t* sA = smem + kOffA;  // K tiles
  uint8_t* sB = smem + kOffB;  // V tiles
  volatile int32_t* abort = &bar->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int per = p.hq * p.B;
  const int qt = p.nq - 1 - u / per;  // longest rows first
  const int h = (u % per) % p.hq, b = (u % per) / p.hq;
  const int hk = h / (p.hq / p.hkv);
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, false);
  const int32_t q0r = qt * kT, q1r = min(p.S, q0r + kT) - 1;
  const int64_t q0 = (int64_t)c0 + q0r, q1 = (int64_t)c0 + q1r;
  // key tiles that can hold an admitted pair (the forward's): prefix tiles, then the band
  const int32_t kc = keys_below(km, q1 + 1);
  const int32_t kP = keys_below(km, P);
  const int t1_end = (min(kP, kc) + kT - 1) / kT;
  const int32_t kw = keys_below(km, q0 - p.W + 1);
  const int t2_begin = max(t1_end, kw / kT);
  const int t2_end = (kc + kT - 1) / kT;
  const int n = t1_end + max(0, t2_end - t2_begin);
  auto tile_at = [&](int i) { return i < t1_end ? i : t2_begin + (i - t1_end); };

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&p.tmq);
      prefetch_tmap(&p.tmdo);
      prefetch_tmap(&p.tmk);
      prefetch_tmap(&p.tmv);
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(&bar->res_full, 2 * kB);
      for (int x = 0; x < kNH; ++x) {
        tma_load_4d(sQ + x * kHalf, &p.tmq, &bar->res_full, 64 * x, h, q0r, b, pol_q);
        tma_load_4d(sdO + x * kHalf, &p.tmdo, &bar->res_full, 64 * x, h, q0r, b, pol_q);
      }
      fl.res = 1;
      for (int t = 0; t < n; ++t) {
        const int ka = tile_at(t) * kT;
        const int sa = t % kSa, sb = t % kSb;
        if (!mbar_wait_abort(&bar->a_empty[sa], ((t / kSa) & 1) ^ 1, abort, p.wait_ns)) break;
        uint64_t* fa = &bar->a_full[sa];
        mbar_arrive_expect_tx(fa, kB);
        for (int x = 0; x < kNH; ++x)
          tma_load_4d(sA + sa * kTile + x * kHalf, &p.tmk, fa, 64 * x, hk, ka, b, pol_kv);
        fl.a[sa] = (t / kSa) & 1;
        if (!mbar_wait_abort(&bar->b_empty[sb], ((t / kSb) & 1) ^ 1, abort, p.wait_ns)) break;
        uint64_t* fb = &bar->b_full[sb];
        mbar_arrive_expect_tx(fb, kB);
        for (int x = 0; x < kNH; ++x)
          tma_load_4d(sB + sb * kTile + x * kHalf, &p.tmv, fb, 64 * x, hk, ka, b, pol_kv);
        fl.b[sb] = (t / kSb) & 1;
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint64_t aQ = tc::sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t aO = tc::sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t bK = tc::sdesc_sw128(smem_u32(sA), 16, 1024);       // K-major
      const uint64_t bKm = tc::sdesc_sw128(smem_u32(sA), kHalf, 1024);   // MN-major
      const uint64_t bV = tc::sdesc_sw128(smem_u32(sB), 16, 1024);
      auto soa = [](int t) { return (uint64_t)(((t % kSa) * kTile) >> 4); };
      auto sob = [](int t) { return (uint64_t)(((t % kSb) * kTile) >> 4); };
      // per step t (buffer t & 1): dP = dO V^T, then S of step t+1, then dQ += dS K
      bool ok = mbar_wait_abort(&bar->res_full, 0, abort, p.wait_ns) &&
                mbar_wait_abort(&bar->a_full[0], 0, abort, p.wait_ns);
      if (ok) {
        tc::fence_after();
        mma_ss8<D>(tmem, aQ, bK + soa(0), false);  // S(0) = Q K(0)^T
        tc::commit(smem_u32(&bar->s_full[0]));
      }
      for (int t = 0; ok && t < n; ++t) {
        const int bf = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        const uint32_t tb = tmem + bf * 128;
        if (!(ok = mbar_wait_abort(&bar->p_ready[bf], ph, abort, p.wait_ns) &&
                   mbar_wait_abort(&bar->b_full[t % kSb], (t / kSb) & 1, abort, p.wait_ns)))
          break;
        tc::fence_after();
        mma_ss8<D>(tb, aO, bV + sob(t), false);  // dP = dO V^T
        tc::commit(smem_u32(&bar->dp_full[bf]));
        tc::commit(smem_u32(&bar->b_empty[t % kSb]));
        if (t + 1 < n) {
          if (!(ok = mbar_wait_abort(&bar->a_full[(t + 1) % kSa], ((t + 1) / kSa) & 1, abort, p.wait_ns)))
            break;
          tc::fence_after();
          mma_ss8<D>(tmem + (bf ^ 1) * 128, aQ, bK + soa(t + 1), false);
          tc::commit(smem_u32(&bar->s_full[bf ^ 1]));
        }
        if (!(ok = mbar_wait_abort(&bar->ds_ready[bf], ph, abort, p.wait_ns))) break;
        tc::fence_after();
        mma_ts8<D>(tmem + kTAcc, tb, bKm + soa(t), t > 0);  // dQ += dS K
        tc::commit(smem_u32(&bar->a_empty[t % kSa]));
      }
      if (ok) tc::commit(smem_u32(&bar->done));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, part = warp >> 2;
    const int row = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t qpos = q0 + row;
    const float2 ldr = p.ld[((int64_t)b * p.hq + h) * p.s_pad + q0r + row];  // rows < s_pad
    // admitted key indices of this row: [0, a1) and [b0, b1)
    const int32_t a1 = keys_below(km, min((int64_t)P, qpos + 1));
    const int32_t b0 = keys_below(km, max((int64_t)0, qpos - p.W + 1));
    const int32_t b1 = keys_below(km, qpos + 1);
    bool ok = true;
    float pr[kNC];
    for (int t = 0; t < n; ++t) {
      const int bf = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      const int32_t ka = tile_at(t) * kT;
      const int32_t kb = min(km.n_keys, ka + kT) - 1;
      const bool masked = ka + kT > km.n_keys ||
                          tile_class(km, c0, q0r, q1r, ka, kb, P, p.W) != kFull;
      const int32_t base = ka + part * kNC;
      const uint32_t tS = tmem + bf * 128 + part * kNC + lane_off;
      uint32_t kmask[kNC / 32];
      if (masked) {
#pragma unroll
        for (int w = 0; w < kNC / 32; ++w)
          kmask[w] = keep_bits(32 * w, a1 - base, b0 - base, b1 - base);
      }
      ok = mbar_wait_abort(&bar->s_full[bf], ph, abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      if (masked)
        p_row<true>(tS, p.scale_log2, ldr.x, kmask, pr);
      else
        p_row<false>(tS, p.scale_log2, ldr.x, kmask, pr);
      release(&bar->p_ready[bf], lane, false);
      ok = mbar_wait_abort(&bar->dp_full[bf], ph, abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      ds_row(tS, ldr.y, pr);
      release(&bar->ds_ready[bf], lane, true);
    }
    if (ok && n > 0) {
      ok = mbar_wait_abort(&bar->done, 0, abort, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc::fence_after();
      const bool valid = q0r + row <= q1r;
      float* dst = p.dq + (((int64_t)b * p.S + (valid ? q0r + row : 0)) * p.hq + h) * D;
      if (n > 0 && D == 128) {
        store_chunk_tma(tmem + kTAcc + lane_off, smem + kOffA + warp * 8192, &p.tmdq, part,
                        p.scale, true, (int32_t)qpos, p.turns, h, q0r + quad * 32, b, lane);
        if (lane == 0) bulk_wait_read_all();
      } else if (n > 0) {
        store_chunk<D>(tmem + kTAcc + lane_off, dst, part, valid, p.scale, true, (int32_t)qpos,
                       p.turns);
      } else if (valid) {
        constexpr int kPairs = Geo<D>::kPairs;
        for (int e = part * kPairs; e < part * kPairs + kPairs; e += 4) {
          *reinterpret_cast<float4*>(dst + e) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dst + D / 2 + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  Bars* bar = reinterpret_cast<Bars*>(smem + kOffBars);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::alloc(smem_u32(&bar->tmem_slot), 512);
    tc::relinquish();
  }
  if (tid == 32) {
    mbar_init(&bar->res_full, 1);
    for (int s = 0; s < kSaQ; ++s) {
      mbar_init(&bar->a_full[s], 1);
      mbar_init(&bar->a_empty[s], 1);
    }
    for (int s = 0; s < kSb; ++s) {
      mbar_init(&bar->b_full[s], 1);
      mbar_init(&bar->b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_ready[i], kSoftWarps);  // one arrival per softmax warp
      mbar_init(&bar->dp_full[i], 1);
      mbar_init(&bar->ds_ready[i], kSoftWarps);
    }
    mbar_init(&bar->done, 1);
    mbar_init(&bar->drain, 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bar->tmem_slot;
  grid_dependency_wait();  // rotated Q / K and the LSE / D pairs come from the pre-pass

  const int u = (int)blockIdx.x;
  Inflight fl;
  fl.res = 0;
  for (int s = 0; s < kSaQ; ++s) fl.a[s] = -1;
  for (int s = 0; s < kSb; ++s) fl.b[s] = -1;
  if (u < p.n_dkdv)
    dkdv_cta<D>(p, smem, bar, tmem, u, fl);
  else
    dq_cta<D>(p, smem, bar, tmem, u - p.n_dkdv, fl);

  tc::fence_before();
  __syncthreads();
  if (bar->abort) {
    // A wait gave up.  Before shared and tensor memory are released, everything
    // issued must have landed: the producer waits (bounded) for the last load
    // into each slot -- a completed phase answers at once, and no later phase
    // can complete now -- and the issuer commits once more and waits until all
    // its products have completed.
    if (tid == 0) set_flag(p.status, PS_DEV_TIMEOUT);
    const int lane = tid & 31;
    if (warp == kProducerWarp && lane == 0) {
      if (fl.res) mbar_wait(&bar->res_full, 0, p.wait_ns);
      for (int s = 0; s < kSaQ; ++s)
        if (fl.a[s] >= 0) mbar_wait(&bar->a_full[s], (uint32_t)fl.a[s], p.wait_ns);
      for (int s = 0; s < kSb; ++s)
        if (fl.b[s] >= 0) mbar_wait(&bar->b_full[s], (uint32_t)fl.b[s], p.wait_ns);
    } else if (warp == kMmaWarp && lane == 0) {
      tc::commit(smem_u32(&bar->drain));
      mbar_wait(&bar->drain, 0, p.wait_ns);
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
  L.s_pad = (S + kT - 1) / kT * kT;
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
  if (head_dim != 64 && head_dim != 128) return PS_ERR_UNSUPPORTED;
  *bytes = bwd::layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim).total;
  return PS_OK;
}

extern "C" ps_status_t ps_prefill_backward(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* d_out,
                                           int32_t batch, int32_t seqlen, const int32_t* q_start,
                                           const int32_t* prefix_len, int32_t window,
                                           int32_t n_q_heads, int32_t n_kv_heads,
                                           int32_t head_dim, float scale, double rope_theta,
                                           const void* fwd_workspace, float* dq, float* dk,
                                           float* dv, void* workspace, size_t workspace_bytes,
                                           int32_t* status, void* stream) {
  if (!q || !k || !v || !out || !lse || !d_out || !q_start || !prefix_len || !dq || !dk || !dv)
    return PS_ERR_INVALID_ARGUMENT;
  if (batch < 1 || seqlen < 1 || window < 1 || n_q_heads < 1 || n_kv_heads < 1 ||
      n_q_heads % n_kv_heads || !(scale > 0.f) || !(rope_theta > 0.0))
    return PS_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return PS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(d_out) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return PS_ERR_ALIGNMENT;
  const bwd::Layout L = bwd::layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PS_ERR_WORKSPACE;
  if (workspace_bytes < L.total) return PS_ERR_WORKSPACE;
  if (fwd_workspace && (reinterpret_cast<uintptr_t>(fwd_workspace) & 255u)) return PS_ERR_WORKSPACE;
  const int32_t nq = (seqlen + bwd::kT - 1) / bwd::kT;
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
  // rotated Q and K: the forward's (same layout at the start of its workspace),
  // or rotated here into this workspace
  const uint8_t* qk = fwd_workspace ? static_cast<const uint8_t*>(fwd_workspace) : ws;
  g.qh = reinterpret_cast<uint4*>(ws + L.q_off);
  g.kh = reinterpret_cast<uint4*>(ws + L.k_off);
  g.rotate = fwd_workspace ? 0 : 1;
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
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
    const int64_t blocks = groups < cap ? groups : cap;
    if (launch_dependent(head_dim == 128 ? bwd::bwd_prep_kernel<128> : bwd::bwd_prep_kernel<64>,
                         dim3((unsigned)blocks), dim3(256), 0, s, g) != cudaSuccess)
      return PS_ERR_CUDA;
  }

  bwd::Params p;
  const uint64_t qd[4] = {(uint64_t)head_dim, (uint64_t)n_q_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t qs[3] = {(uint64_t)head_dim * 2, (uint64_t)n_q_heads * head_dim * 2,
                          (uint64_t)seqlen * n_q_heads * head_dim * 2};
  const uint64_t kd[4] = {(uint64_t)head_dim, (uint64_t)n_kv_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t ks[3] = {(uint64_t)head_dim * 2, (uint64_t)n_kv_heads * head_dim * 2,
                          (uint64_t)seqlen * n_kv_heads * head_dim * 2};
  const uint32_t box[4] = {64u, 1u, (uint32_t)bwd::kT, 1u};
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool okm = encode_tmap(&p.tmq, bf, 4, qk + L.q_off, qd, qs, box, sw) &&
                   encode_tmap(&p.tmdo, bf, 4, d_out, qd, qs, box, sw) &&
                   encode_tmap(&p.tmk, bf, 4, qk + L.k_off, kd, ks, box, sw) &&
                   encode_tmap(&p.tmv, bf, 4, v, kd, ks, box, sw);
  if (!okm) return PS_ERR_CUDA;
  if (head_dim == 128) {
    const uint64_t fqs[3] = {(uint64_t)head_dim * 4, (uint64_t)n_q_heads * head_dim * 4,
                             (uint64_t)seqlen * n_q_heads * head_dim * 4};
    const uint64_t fks[3] = {(uint64_t)head_dim * 4, (uint64_t)n_kv_heads * head_dim * 4,
                             (uint64_t)seqlen * n_kv_heads * head_dim * 4};
    const uint32_t fbox[4] = {32u, 1u, 32u, 1u};
    const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (!encode_tmap(&p.tmdq, f32, 4, dq, qd, fqs, fbox, sw) ||
        !encode_tmap(&p.tmdk, f32, 4, dk, kd, fks, fbox, sw) ||
        !encode_tmap(&p.tmdv, f32, 4, dv, kd, fks, fbox, sw))
      return PS_ERR_CUDA;
  }
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
  const WaitHooks hooks = wait_hooks();
  p.wait_ns = hooks.wait_ns;
  p.drop_first_load = hooks.drop_first_load;
  make_rope_turns(rope_theta, head_dim, &p.turns);
  auto kern = head_dim == 128 ? bwd::bwd_kernel<128> : bwd::bwd_kernel<64>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bwd::kSmem) !=
      cudaSuccess)
    return PS_ERR_CUDA;
  if (launch_dependent(kern, dim3((unsigned)(n_dkdv + n_dq)), dim3(bwd::kThreads),
                       (size_t)bwd::kSmem, s, p) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}
