// ps_prefill.cu -- Prefix-Sliding prefill / extend / training forward.
//
// Two kernels per call:
//  1. rope_gather_kernel rotates Q and the chunk's K at their absolute
//     positions (Continue PE) into the workspace; with a ring it first copies
//     the ring's live keys and values (already rotated when appended) in
//     position order, so the key array is [cached prefix][cached window][chunk].
//  2. the tile kernel: prefill_pair_kernel (warp-specialised, two query heads
//     of one KV head per CTA) when the GQA group size is even, else
//     prefill_kernel: one CTA per (128-query tile, query head, batch row).  It
//     visits only the key tiles that can hold an admitted pair -- the prefix
//     tiles and the band of tiles around the diagonal -- and classifies each:
//     FULL tiles run unmasked, PARTIAL tiles get the element mask ("Prefix
//     Sliding for efficient test-time scaling", agihunt.info, paragraph on the
//     kernel's two-level filter).  S = Q K^T and O += P V run on tcgen05 tensor
//     cores with fp32 accumulators in TMEM; softmax runs one thread per query
//     row straight out of TMEM.
#include "ps_internal.h"
#include "ps_math.cuh"
#include "ps_tc.cuh"
#include "ps_rope.cuh"
#include "ps_tiles.cuh"

namespace ps {

// ---------------------------------------------------------------------------
// tile export
// ---------------------------------------------------------------------------
__global__ void tile_classes_kernel(KeyMap m, int32_t seqlen, int32_t q_start, int32_t P,
                                    int32_t W, int32_t bm, int32_t bn, int32_t nq, int32_t nk,
                                    uint8_t* __restrict__ out) {
  const int64_t n = (int64_t)nq * nk;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int a = (int)(i / nk), b = (int)(i % nk);
    const int32_t qa = a * bm, qb = min(seqlen, (a + 1) * bm) - 1;
    const int32_t ka = b * bn, kb = min(m.n_keys, (b + 1) * bn) - 1;
    out[i] = tile_class(m, q_start, qa, qb, ka, kb, P, W);
  }
}

// ---------------------------------------------------------------------------
// 1. RoPE + gather
// ---------------------------------------------------------------------------
struct GatherParams {
  const uint4* q;  // [B, S, Hq, D]
  const uint4* k;  // [B, S, Hkv, D]
  const uint4* v;
  uint4* qh;       // [B, S, Hq, D]       rotated
  uint4* qr;       // [B, S, Hq, D]       rotated at the Reset PE position, or null
  uint4* kh;       // [B, Skv, Hkv, D]    rotated (ring part gathered)
  uint4* vg;       // [B, Skv, Hkv, D]    gathered values (ring only) or null
  const int32_t* q_start;
  const int32_t* prefix_len;
  int32_t* status;
  // ring (null k_pool = no ring)
  const uint4* k_pool;
  const uint4* v_pool;
  const int32_t* ring_prefix;
  const int32_t* ring_seq;
  SlotMap map;
  int32_t nseq;
  int32_t B, S, Skv, hq, hkv, W;
  RopeTurns turns;
};

constexpr int kRopeRows = 8;  // chunk rows per block iteration
constexpr int kRopeBatch = 4; // items a thread loads before it rotates and stores any

// D = 64 or 128.  Phase A: groups of kRopeRows chunk rows; the D/2 (cos, sin)
// pairs of each row's position are computed once into shared memory and shared
// by all Hq query heads and Hkv key heads of that row.  Under Reset PE the query is
// also rotated at min(p, P + W - 1), its position once the cache is renumbered
// (prefix keys keep theirs), into qr.  Each thread then loads
// kRopeBatch items (8 rotation pairs of one row and head each) before it
// rotates and stores them, to keep enough loads in flight.  Phase B: the ring
// rows (copied, already rotated) and the zero padding of each batch row's key
// array.
// RESET: also write qr (a separate instance keeps the other's registers down).
template <bool RESET, int D>
__global__ void __launch_bounds__(256) rope_gather_kernel(const __grid_constant__ GatherParams p) {
  constexpr int VEC = D / 8, HALFV = D / 16, NPAIR = D / 2, NG = D / 16;  // NG groups of 8 pairs
  __shared__ float2 cs[kRopeRows][NPAIR];
  __shared__ float2 csr[RESET ? kRopeRows : 1][NPAIR];  // Reset PE query angles
  grid_dependency_wait();  // inputs and workspace may be in use by earlier stream work
  allow_dependents();      // the tile kernel may set up meanwhile; it waits for this one
  const bool ring = p.k_pool != nullptr;
  const int64_t n_rows = (int64_t)p.B * p.S;
  const int64_t n_groups = (n_rows + kRopeRows - 1) / kRopeRows;
  const int heads = p.hq + p.hkv;
  for (int64_t grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
    const int64_t r0 = grp * kRopeRows;
    for (int x = threadIdx.x; x < kRopeRows * NPAIR; x += blockDim.x) {
      const int rr = x / NPAIR, i = x % NPAIR;
      const int64_t r = r0 + rr;
      if (r < n_rows) {
        const int b = (int)(r / p.S);
        const int32_t pos = p.q_start[b] + (int32_t)(r % p.S);
        float c, sn;
        rope_cos_sin(pos, p.turns.f[i], c, sn);
        cs[rr][i] = make_float2(c, sn);
        if (RESET) {
          const int64_t last = (int64_t)p.prefix_len[b] + p.W - 1;  // renumbered position cap
          if ((int64_t)pos > last && last >= 0) rope_cos_sin((int32_t)last, p.turns.f[i], c, sn);
          csr[rr][i] = make_float2(c, sn);
        }
      }
    }
    __syncthreads();
    const int items = kRopeRows * heads * NG;
    for (int it0 = threadIdx.x; it0 < items; it0 += kRopeBatch * blockDim.x) {
      uint4 xa[kRopeBatch], xb[kRopeBatch];
      uint4* dst[kRopeBatch];
      uint4* dstr[kRopeBatch];
      const float2* ang[kRopeBatch];
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        dst[u] = nullptr;
        dstr[u] = nullptr;
        const int it = it0 + u * blockDim.x;
        if (it >= items) continue;
        const int g = it % NG;
        const int hd = (it / NG) % heads;
        const int rr = (it / NG) / heads;
        const int64_t r = r0 + rr;
        if (r >= n_rows) continue;
        ang[u] = &cs[rr][8 * g];
        if (hd < p.hq) {
          const int64_t base = (r * p.hq + hd) * VEC + g;
          xa[u] = p.q[base];
          xb[u] = p.q[base + HALFV];
          dst[u] = p.qh + base;
          if (RESET) dstr[u] = p.qr + base;
        } else {
          const int h = hd - p.hq;
          const int b = (int)(r / p.S);
          const int32_t t = (int32_t)(r % p.S);
          const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
          const KeyMap km = make_keymap(p.S, c0, P, p.W, ring);
          const int32_t n_ring = km.n_keys - p.S;
          // the ring part must fit the workspace stride: 0 <= P <= the ring's
          // prefix_max (which ps_prefill sized it by) and q_start >= 0
          if (c0 < 0 || (ring && (P < 0 || n_ring > p.Skv - p.S))) {
            set_flag(p.status, c0 < 0 ? PS_DEV_BAD_POS : PS_DEV_BAD_PREFIX);
            continue;
          }
          const int64_t src = (r * p.hkv + h) * VEC + g;
          const int64_t d = (((int64_t)b * p.Skv + n_ring + t) * p.hkv + h) * VEC + g;
          xa[u] = p.k[src];
          xb[u] = p.k[src + HALFV];
          dst[u] = p.kh + d;
          if (p.vg) {
            p.vg[d] = p.v[src];
            p.vg[d + HALFV] = p.v[src + HALFV];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        if (!dst[u]) continue;
        uint4 ra, rb;
        rotate8(xa[u], xb[u], ang[u], ra, rb);
        dst[u][0] = ra;
        dst[u][HALFV] = rb;
        if (RESET && dstr[u]) {
          const float2* angr = &csr[0][0] + (ang[u] - &cs[0][0]);
          rotate8(xa[u], xb[u], angr, ra, rb);
          dstr[u][0] = ra;
          dstr[u][HALFV] = rb;
        }
      }
    }
    __syncthreads();
  }

  // phase B: per batch row, key indices [0, n_ring) come from the ring and
  // [n_keys, Skv) are padding up to the workspace stride
  const int32_t extra = p.Skv - p.S;
  const int64_t n_extra = (int64_t)p.B * extra * p.hkv * VEC;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < n_extra;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int vec = (int)(u % VEC);
    int64_t rest = u / VEC;
    const int h = (int)(rest % p.hkv);
    rest /= p.hkv;
    const int b = (int)(rest / extra);
    const int32_t x = (int32_t)(rest % extra);
    const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
    const KeyMap km = make_keymap(p.S, c0, P, p.W, ring);
    const int32_t n_ring = km.n_keys - p.S;
    const int32_t kidx = x < n_ring ? x : x + p.S;
    const int64_t dst = (((int64_t)b * p.Skv + kidx) * p.hkv + h) * VEC + vec;
    uint4 kk = make_uint4(0, 0, 0, 0), vv = kk;
    if (kidx < km.n_keys) {  // cached key: copy the rotated row out of the ring
      const int32_t s = p.ring_seq ? p.ring_seq[b] : b;
      bool bad = s < 0 || s >= p.nseq;
      if (bad) {
        set_flag(p.status, PS_DEV_BAD_SEQ);
      } else {
        if (p.ring_prefix[s] != P) { set_flag(p.status, PS_DEV_BAD_PREFIX); bad = true; }
        if (!p.map.seq_ok(s)) { set_flag(p.status, PS_DEV_BAD_SLOT); bad = true; }
        if (!bad) {
          const int32_t pos = key_pos(km, kidx);
          const int64_t r = p.map.row(s, ring_slot(pos, P, p.W));
          if (r < 0) {
            set_flag(p.status, PS_DEV_BAD_SLOT);
          } else {
            const int64_t src = (r * p.hkv + h) * VEC + vec;
            kk = p.k_pool[src];
            vv = p.v_pool[src];
          }
        }
      }
    }
    p.kh[dst] = kk;
    if (p.vg) p.vg[dst] = vv;
  }
}

// ---------------------------------------------------------------------------
// 2. tile kernel
// ---------------------------------------------------------------------------
constexpr int kBM = 128, kBN = 128;
constexpr int kHalf = kBM * 64 * 2;  // one 64-column swizzled half block: 16 KB
constexpr int kPTile = 2 * kHalf;    // 128 x 128 bf16 probabilities: 32 KB
constexpr uint32_t kIdescQK = tc::idesc_bf16(kBM, kBN, false);

// Q, K and V tiles of 128 rows for head dim D (64 or 128): D / 64 half blocks.
template <int D>
struct Geom {
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kIdescPV = tc::idesc_bf16(kBM, D, true);
  static constexpr int kSmemSingle = 5 * kTile + kPTile + 1024 /*barriers*/ + 1024 /*alignment*/;
};

struct PrefillParams {
  CUtensorMap tmq;  // rotated Q  {D, Hq, S, B}
  CUtensorMap tmqr; // Q rotated at the Reset PE position (same layout); unused otherwise
  CUtensorMap tmk;  // rotated K  {D, Hkv, Skv, B}
  CUtensorMap tmv;  // values     {D, Hkv, S or Skv, B}
  __nv_bfloat16* out;
  float* lse;
  int32_t out32;  // out is 32-byte aligned: rows are stored 32 bytes at a time
  const int32_t* q_start;
  const int32_t* prefix_len;
  int32_t* status;
  int32_t S, hq, hkv, W, with_ring, nq, B;
  int32_t reset;  // Reset PE: prefix keys are scored with the tmqr query
  float scale_log2;
  uint64_t wait_ns;          // bounded-wait limit
  int32_t drop_first_load;   // test hook: CTA 0 skips its first K/V copy
};

// The key tiles one 128-row query tile visits, in order: the tiles that hold
// prefix keys, [0, t1_end), then the band of tiles that can hold window keys of
// some row, [t2_begin, t2_end); tiles in neither hold no admitted pair.
//
// Reset PE (agihunt.info paragraph on position encodings; the renumbering is
// the one ps_decode uses): the cache is renumbered for each query, prefix keys
// keep their positions, the window keys follow them in order and the query at
// absolute position p becomes the newest entry, min(p, P + W - 1).  Window keys
// keep their distance to the query; prefix keys see the query rotated at
// min(p, P + W - 1) instead of p, which differs only for rows p > P + W - 1.
// For a tile with such rows the prefix tiles are visited with that second
// query ("renumbered visits", [0, n0)); if one tile holds both the last prefix
// key and later keys that some row admits, it is visited twice: first for its
// prefix keys (renumbered query), then for its later keys (absolute query).
enum : int { kVisitAll = 0, kVisitPrefixPart = 1, kVisitLaterPart = 2 };

struct Visits {
  int t1_end, t2_begin, n;  // n = visits
  int n0;                   // visits [0, n0) use the renumbered query
  int ts;                   // visit of the split tile's prefix part, or -1
  int32_t kP;               // keys with position < P

  __device__ __forceinline__ int tile(int j) const {
    if (ts < 0) return j < t1_end ? j : t2_begin + (j - t1_end);
    if (j <= ts) return j;
    return j == ts + 1 ? ts : t2_begin + (j - t1_end - 1);
  }
  __device__ __forceinline__ int mode(int j) const {
    if (ts < 0) return kVisitAll;
    return j == ts ? kVisitPrefixPart : (j == ts + 1 ? kVisitLaterPart : kVisitAll);
  }
};

__device__ __forceinline__ Visits make_visits(const KeyMap& km, int64_t q0, int64_t q1, int32_t P,
                                              int32_t W, bool reset) {
  Visits v;
  const int32_t kc = keys_below(km, q1 + 1);  // keys at or before the last query
  v.kP = keys_below(km, P);                   // prefix keys
  v.t1_end = (min(v.kP, kc) + kBN - 1) / kBN;
  const int32_t kw = keys_below(km, q0 - W + 1);
  v.t2_begin = max(v.t1_end, kw / kBN);
  const int t2_end = (kc + kBN - 1) / kBN;
  v.n = v.t1_end + max(0, t2_end - v.t2_begin);
  v.n0 = 0;
  v.ts = -1;
  if (reset && v.kP > 0 && q1 > (int64_t)P + W - 1) {
    // here kc >= kP, so tiles [0, t1_end) hold exactly the prefix keys
    v.n0 = v.t1_end;
    if (v.kP % kBN) {
      const int32_t ka = v.kP, kb = min(km.n_keys, v.t1_end * kBN) - 1;
      if (kb >= ka && interval_any(q0, q1, key_pos(km, ka), key_pos(km, kb), P, W)) {
        v.ts = v.t1_end - 1;
        v.n += 1;
      }
    }
  }
  return v;
}

// 32 fp32 columns of one output row (O * inv) as bf16 at dst.  One lane writes
// one row, so each store instruction touches 32 rows: 32-byte pieces (dst
// 32-byte aligned, out32) fill whole sectors, with half as many instructions as
// 16-byte ones.
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* dst, const uint32_t (&o)[32],
                                                float inv, bool out32) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    w[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
  if (out32) {
#pragma unroll
    for (int e = 0; e < 16; e += 8)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 2 * e),
                   "r"(w[e]), "r"(w[e + 1]), "r"(w[e + 2]), "r"(w[e + 3]), "r"(w[e + 4]),
                   "r"(w[e + 5]), "r"(w[e + 6]), "r"(w[e + 7])
                   : "memory");
  } else {
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      *reinterpret_cast<uint4*>(dst + 2 * e) = make_uint4(w[e], w[e + 1], w[e + 2], w[e + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(128, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int kTile = Geom<D>::kTile, kHalves = Geom<D>::kHalves;
  constexpr uint32_t kIdescPV = Geom<D>::kIdescPV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sK0 = smem + kTile;
  uint8_t* sV0 = smem + 3 * kTile;
  uint8_t* sP = smem + 5 * kTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + kPTile);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;  // [2]
  uint64_t* s_done = bars + 3;
  uint64_t* o_done = bars + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = p.nq - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.hq / p.hkv);
  const int32_t c0 = p.q_start[b], P = p.prefix_len[b];
  const KeyMap km = make_keymap(p.S, c0, P, p.W, p.with_ring != 0);
  const int32_t q0r = qt * kBM, q1r = min(p.S, q0r + kBM) - 1;
  const int64_t q0 = (int64_t)c0 + q0r, q1 = (int64_t)c0 + q1r;

  // key tiles that can hold an admitted pair: the prefix tiles, then the band
  const Visits vs = make_visits(km, q0, q1, P, p.W, p.reset != 0);
  const int n_tiles = vs.n;
  auto tile_at = [&](int it) { return vs.tile(it); };

  if (warp == 0) {
    tc::alloc(smem_u32(tmem_slot), 256);
    tc::relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    prefetch_tmap(&p.tmq);
    prefetch_tmap(&p.tmk);
    prefetch_tmap(&p.tmv);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;
  grid_dependency_wait();  // rotated Q / K come from the pre-pass
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  // test hook: CTA (0, 0, 0) skips its first K / V copy and arrival
  const int dropped = p.drop_first_load && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0
                          ? 0 : -1;
  int load_no = 0;
  auto load_kv = [&](int stage, int kt) {
    if (load_no++ == dropped) return;
    uint8_t* dk = sK0 + stage * kTile;
    uint8_t* dv = sV0 + stage * kTile;
    mbar_arrive_expect_tx(&kv_full[stage], 2 * kTile);
    for (int hh = 0; hh < kHalves; ++hh) {
      tma_load_4d(dk + hh * kHalf, &p.tmk, &kv_full[stage], 64 * hh, hk, kt * kBN, b, pol_kv);
      tma_load_4d(dv + hh * kHalf, &p.tmv, &kv_full[stage], 64 * hh, hk, kt * kBN, b, pol_kv);
    }
  };
  int issued = 0;  // key tiles whose loads were issued (thread 0)
  int q_pending = -1;  // parity of a Q load issued but not yet waited for (thread 0)
  auto load_q = [&](const CUtensorMap* m, int parity) {
    mbar_arrive_expect_tx(q_full, kTile);
    for (int hh = 0; hh < kHalves; ++hh)
      tma_load_4d(sQ + hh * kHalf, m, q_full, 64 * hh, h, q0r, b, pol_q);
    q_pending = parity;
  };
  if (tid == 0 && n_tiles > 0) {
    load_q(vs.n0 > 0 ? &p.tmqr : &p.tmq, 0);  // Reset PE: renumbered query first
    for (; issued < 2 && issued < n_tiles; ++issued) load_kv(issued, tile_at(issued));
  }

  const int row = tid;
  const int64_t qpos = q0 + row;
  // admitted key indices of this row: [0, a1) and [b0, b1)
  const int32_t a1 = keys_below(km, min((int64_t)P, qpos + 1));
  const int32_t b0 = keys_below(km, max((int64_t)0, qpos - p.W + 1));
  const int32_t b1 = keys_below(km, qpos + 1);
  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;
  int committed_pv = 0;
  int it = 0;
  for (; it < n_tiles; ++it) {
    const int st = it & 1;
    const int kt = tile_at(it);
    const int32_t ka = kt * kBN;
    const int32_t kb = min(km.n_keys, ka + kBN) - 1;
    const uint8_t cls = tile_class(km, c0, q0r, q1r, ka, kb, P, p.W);
    const int mode = vs.mode(it);
    const bool masked = cls != kFull || ka + kBN > km.n_keys || mode != kVisitAll;

    if (tid == 0) {
      bool w = true;
      // Reset PE: after the renumbered visits the query at its own position
      // replaces the renumbered one (every Q K reading sQ has completed)
      if (it > 0 && it == vs.n0) load_q(&p.tmq, 1);
      if (it == 0 || it == vs.n0) {
        w = mbar_wait(q_full, q_pending, p.wait_ns);
        if (w) q_pending = -1;
      }
      w = w && mbar_wait(&kv_full[st], (it >> 1) & 1, p.wait_ns);
      if (w) {
        tc::fence_after();
        const uint32_t aq = smem_u32(sQ), ak = smem_u32(sK0 + st * kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tS, tc::sdesc_sw128(aq + off, 16, 1024), tc::sdesc_sw128(ak + off, 16, 1024),
                       kIdescQK, kk > 0);
        }
      } else {
        ok = false;
      }
      tc::commit(smem_u32(s_done));  // arrives at once if nothing was issued
    }
    if (!mbar_wait(s_done, it & 1, p.wait_ns)) ok = false;
    // tcgen05.ld / st are warp-collective (.sync.aligned): reconverge after the
    // per-thread spin above before touching tensor memory
    __syncwarp();
    tc::fence_after();

    // ---- scores of this thread's query row
    float s[kBN];
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      tc::ld32(tS + lane_off + c * 32, r);
      tc::wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) s[c * 32 + j] = __uint_as_float(r[j]) * p.scale_log2;
    }
    if (masked) {
      // kept columns: j < A1 (prefix keys) or B0 <= j < B1 (window keys); a
      // split tile's two visits keep only the keys before / after the prefix
      const int32_t A1 = mode == kVisitLaterPart ? 0 : a1 - ka;
      const int32_t B0 =
          mode == kVisitPrefixPart ? 0 : (mode == kVisitLaterPart ? max(b0, vs.kP) : b0) - ka;
      const int32_t B1 = mode == kVisitPrefixPart ? 0 : b1 - ka;
      uint32_t kmask[kBN / 32];
#pragma unroll
      for (int w = 0; w < kBN / 32; ++w) kmask[w] = keep_bits(32 * w, A1, B0, B1);
#pragma unroll
      for (int j = 0; j < kBN; ++j) s[j] = (kmask[j >> 5] & (1u << (j & 31))) ? s[j] : -INFINITY;
    }
    float mt = s[0];
#pragma unroll
    for (int j = 1; j < kBN; ++j) mt = fmaxf(mt, s[j]);
    const float m_new = fmaxf(m_ref, mt);
    float alpha = 1.f;
    bool rescale = false;
    if (it == 0) {
      m_ref = m_new;  // the first P V overwrites O
    } else if (m_new > m_ref + 8.f) {  // lazy rescale: keep the stale max while within 2^8
      alpha = ex2(m_ref - m_new);
      m_ref = m_new;
      rescale = true;
    }
    const float mu = m_ref == -INFINITY ? 0.f : m_ref;

    // ---- the previous P V must be done before P and O are touched
    if (it > 0) {
      if (!mbar_wait(o_done, (it - 1) & 1, p.wait_ns)) ok = false;
      tc::fence_after();
      if (tid == 0 && ok && issued < n_tiles) {  // its K/V stage is free: prefetch
        fence_proxy_async_smem();
        load_kv(issued & 1, tile_at(issued));
        ++issued;
      }
    }
    __syncwarp();
    if (__any_sync(0xffffffffu, rescale)) {  // warp-uniform: alpha is 1 on the other rows
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tc::ld32(tO + lane_off + c * 32, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
        tc::st32(tO + lane_off + c * 32, r);
      }
      tc::wait_st();
    }
    // ---- P = exp2(s - m) as bf16 into shared memory, K-major 128-byte
    // swizzle (the A operand of P V), 8 keys (one 16-byte chunk) at a time
    float rs = 0.f;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int j = hh * 64 + c * 8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = ex2(s[j + 2 * e] - mu), bb = ex2(s[j + 2 * e + 1] - mu);
          rs += a + bb;
          w[e] = pack_bf16(a, bb);
        }
        const uint32_t addr = smem_u32(sP) + hh * kHalf + (row >> 3) * 1024 + (row & 7) * 128 +
                              ((c ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
      }
    }
    l = l * alpha + rs;
    fence_proxy_async_smem();
    tc::fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    if (tid == 0) {
      tc::fence_after();
      const uint32_t ap = smem_u32(sP), av = smem_u32(sV0 + st * kTile);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;
        // V is MN-major: 64-column atoms 16 KB apart (LBO), 8-key groups 1 KB apart (SBO)
        tc::mma_bf16(tO, tc::sdesc_sw128(ap + aoff, 16, 1024),
                     tc::sdesc_sw128(av + kk * 2048, kHalf, 1024), kIdescPV, (it > 0) || (kk > 0));
      }
      tc::commit(smem_u32(o_done));
    }
    committed_pv = it + 1;
  }

  if (ok && n_tiles > 0) {
    if (!mbar_wait(o_done, (n_tiles - 1) & 1, p.wait_ns)) ok = false;
    tc::fence_after();
  }
  ok = __all_sync(0xffffffffu, ok);
  if (ok && n_tiles > 0) {
    const float inv = 1.f / l;
    const int32_t qrow = q0r + row;
    __nv_bfloat16* orow = p.out + (((int64_t)b * p.S + qrow) * p.hq + h) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tc::ld32(tO + lane_off + c * 32, r);
      tc::wait_ld();
      if (qrow <= q1r) store_row_chunk(orow + c * 32, r, inv, p.out32 != 0);
    }
    if (qrow <= q1r)
      p.lse[((int64_t)b * p.hq + h) * p.S + qrow] = (m_ref + __log2f(l)) * 0.69314718055994530942f;
  }
  if (!ok && tid == 0) {
    set_flag(p.status, PS_DEV_TIMEOUT);
    // let what was issued land before the CTA's shared memory goes away (bounded)
    for (int t = it; t < issued; ++t)
      if (t != dropped) mbar_wait(&kv_full[t & 1], (t >> 1) & 1, p.wait_ns);
    if (q_pending >= 0) mbar_wait(q_full, q_pending, p.wait_ns);
    if (committed_pv > 0) mbar_wait(o_done, (committed_pv - 1) & 1, p.wait_ns);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// 3. warp-specialised, persistent tile kernel for pairs of query heads that
//    share one KV head (the GQA group size is even).
//
// A work item is one 128-row query tile of two query heads of one batch row.
// Both heads admit the same (query, key) pairs, so they walk the same key
// tiles and every K/V tile staged in shared memory feeds two 128x128
// products.  One CTA per SM walks the items longest-first in a static
// round-robin.  Roles:
//   warps 0-3  softmax, rescale and epilogue of head 0 (one thread per row)
//   warps 4-7  the same for head 1
//   warp 8     TMA producer (Q per item, then K / V tiles through two rings)
//   warps 9-10 tcgen05 issuers, one per head, taking turns
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 columns each.  Each softmax
// thread writes its row of probabilities as bf16 over the first 64 columns of
// its S, and P V reads them from there (tensor-memory A operand), so P never
// touches shared memory.  The products reach the tensor pipe with the heads
// interleaved: P_0 V, S_0 = Q_0 K, P_1 V, S_1 = Q_1 K, so one head's softmax
// overlaps the other head's MMAs.  Each head's products come from its own
// issuing thread, and the two threads pass a token after each group of
// products, so each one's barrier waits run while the other's products
// execute.  Tensor-core instructions of one thread run in issue order, which is
// what lets S_i(j+1) overwrite the columns P_i(j) V has just read.  Across items,
// the next Q is loaded once the last Q K of the current item completes
// (q_empty), and the next item's first P V waits until the epilogue has read
// O out of tensor memory (o_free), so the next item's loads and first Q K
// overlap the current epilogue.  Barrier phases run on across items.
// ---------------------------------------------------------------------------
namespace ws {

constexpr int kThreads = 352;
constexpr int kSt = 2;  // steps in flight: each holds a K tile and a V tile
constexpr int kStK = kSt, kStV = kSt;
template <int D>
constexpr int smem_bytes() {
  return (2 + kStK + kStV) * Geom<D>::kTile + 1024 /*barriers*/ + 1024 /*alignment*/;
}
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // issuers: warps kMmaWarp + head

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t step_full[kSt], step_empty[kSt];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t turn[2];  // turn[i]: issuer i may issue its next group
  uint64_t drain;    // after an abort: the issuers' products have completed
  uint32_t tmem_slot;
  int32_t abort;
};

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort,
                                     uint64_t limit_ns) {
  return mbar_wait_abort(bar, parity, abort, limit_ns);
}

// One work item and the key tiles it visits: the prefix tiles, then the band
// of tiles that can hold window keys of some row of the item.
struct Item {
  int qt, h0, hk, b;
  int32_t c0, P, q0r, q1r;
  int64_t q0, q1;
  KeyMap km;
  Visits v;  // n_tiles = v.n visits
  int n_tiles;
  __device__ __forceinline__ int tile_at(int j) const { return v.tile(j); }
};

__device__ __forceinline__ Item make_item(const PrefillParams& p, int u) {
  Item it;
  const int npairs = p.hq / 2;
  const int per_qt = npairs * p.B;
  it.qt = p.nq - 1 - u / per_qt;  // longest rows first
  const int rem = u % per_qt;
  it.h0 = 2 * (rem % npairs);
  it.b = rem / npairs;
  it.hk = it.h0 / (p.hq / p.hkv);
  it.c0 = p.q_start[it.b];
  it.P = p.prefix_len[it.b];
  it.km = make_keymap(p.S, it.c0, it.P, p.W, p.with_ring != 0);
  it.q0r = it.qt * kBM;
  it.q1r = min(p.S, it.q0r + kBM) - 1;
  it.q0 = (int64_t)it.c0 + it.q0r;
  it.q1 = (int64_t)it.c0 + it.q1r;
  it.v = make_visits(it.km, it.q0, it.q1, it.P, p.W, p.reset != 0);
  it.n_tiles = it.v.n;
  return it;
}

}  // namespace ws

// One query row's share of a 128-key tile: S from TMEM, optional element mask
// (keep column c iff bit c of km is set), online-softmax bookkeeping with a
// lazy rescale, and P = exp2(S * scale - m) stored back over the first 64
// columns as bf16 pairs.  The row sum adds the fp32 probabilities: summing
// the bf16-rounded ones instead moves the LSE of rows with few keys by up to
// a bf16 rounding (2e-3).  Returns the factor O must be scaled by (1 = none).
// The masked and unmasked variants are whole functions so that the 128 scores
// are never live across a branch.  Max, scale and sum use independent chains
// of three-input and packed instructions: this per-row chain, S -> P, is what
// the other head's MMAs have to cover.
template <bool MASK>
__device__ __forceinline__ float softmax_tile(uint32_t tS, int j, float scale_log2,
                                              const uint32_t (&km)[kBN / 32], float& m_used,
                                              float& l) {
  float s[kBN];
  {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tc::ld32(tS, r0);
    tc::ld32(tS + 32, r1);
    tc::ld32(tS + 64, r2);
    tc::ld32(tS + 96, r3);
    tc::wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      s[e] = __uint_as_float(r0[e]);
      s[32 + e] = __uint_as_float(r1[e]);
      s[64 + e] = __uint_as_float(r2[e]);
      s[96 + e] = __uint_as_float(r3[e]);
    }
  }
  if (MASK) {
#pragma unroll
    for (int c = 0; c < kBN; ++c) s[c] = (km[c >> 5] & (1u << (c & 31))) ? s[c] : -INFINITY;
  }
  float mx8[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) mx8[c] = s[c];
#pragma unroll
  for (int c = 8; c < kBN; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], s[c], s[c + 1]);
  const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                         fmaxf(mx8[6], mx8[7]));
  const float m_new = fmaxf(m_used, mx * scale_log2);
  float alpha = 1.f;
  if (j == 0) {
    m_used = m_new;
  } else if (m_new > m_used + 8.f) {  // keep a stale max while within a factor 2^8
    alpha = ex2(m_used - m_new);
    m_used = m_new;
  }
  const float nmu = m_used == -INFINITY ? 0.f : -m_used;
  float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // four packed partial sums
  uint32_t p0[32], p1[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x, y;
    ffma2(x, y, s[2 * c], s[2 * c + 1], scale_log2, scale_log2, nmu, nmu);
    x = ex2(x);
    y = ex2(y);
    p0[c] = pack_bf16(x, y);
    fadd2(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], rs[2 * (c & 3)], rs[2 * (c & 3) + 1], x, y);
  }
  tc::st32(tS, p0);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x, y;
    ffma2(x, y, s[64 + 2 * c], s[64 + 2 * c + 1], scale_log2, scale_log2, nmu, nmu);
    x = ex2(x);
    y = ex2(y);
    p1[c] = pack_bf16(x, y);
    fadd2(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], rs[2 * (c & 3)], rs[2 * (c & 3) + 1], x, y);
  }
  tc::st32(tS + 32, p1);
  l = fmaf(l, alpha, ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7])));
  return alpha;
}

template <int D>
__global__ void __launch_bounds__(ws::kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillParams p) {
  using namespace ws;
  constexpr int kTile = Geom<D>::kTile, kHalves = Geom<D>::kHalves;
  constexpr uint32_t kIdescPV = Geom<D>::kIdescPV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sQ = smem;                   // [2] heads
  uint8_t* sK = smem + 2 * kTile;       // [kStK]
  uint8_t* sV = sK + kStK * kTile;      // [kStV]
  Bars* bar = reinterpret_cast<Bars*>(sV + kStV * kTile);
  volatile int32_t* abort = &bar->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.nq * (p.hq / 2) * p.B;

  if (warp == 0) {
    tc::alloc(smem_u32(&bar->tmem_slot), 512);
    tc::relinquish();
  }
  if (tid == 32) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_empty, 2);  // a commit from each issuer
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&bar->step_full[s], 1);
      mbar_init(&bar->step_empty[s], 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bar->o_done[i], 1);
      mbar_init(&bar->o_free[i], 4);
      mbar_init(&bar->turn[i], 1);
    }
    mbar_init(&bar->drain, 2);
    bar->abort = 0;
    fence_mbar_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bar->tmem_slot;
  grid_dependency_wait();  // rotated Q / K come from the pre-pass
  // What the producer has in flight, for the drain after an abort: the parity of
  // its last Q load and the last step loaded into each stage (-1: none).
  int last_q = -1;
  int last_step[kSt];
#pragma unroll
  for (int s = 0; s < kSt; ++s) last_step[s] = -1;

  // Every role walks the same item sequence; items without tiles (only
  // possible for invalid inputs) are skipped by all of them alike.
  // g counts key tiles and k items processed so far: barrier phases follow them.
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmq);
      prefetch_tmap(&p.tmk);
      prefetch_tmap(&p.tmv);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int g = 0, k = 0, kq = 0;  // kq: Q loads so far (q_full / q_empty phases)
      bool ok = true;
      auto load_q = [&](const Item& it, const CUtensorMap* m) -> bool {
        // every Q K of the previous Q load has completed
        if (!wait(&bar->q_empty, (kq & 1) ^ 1, abort, p.wait_ns)) return false;
        mbar_arrive_expect_tx(&bar->q_full, 2 * kTile);
        for (int i = 0; i < 2; ++i)
          for (int hh = 0; hh < kHalves; ++hh)
            tma_load_4d(sQ + i * kTile + hh * kHalf, m, &bar->q_full, 64 * hh, it.h0 + i, it.q0r,
                        it.b, pol_q);
        last_q = kq & 1;
        ++kq;
        return true;
      };
      for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x) {
        const Item it = make_item(p, u);
        if (it.n_tiles <= 0) continue;
        // Reset PE: the renumbered query serves the first n0 visits
        if (!(ok = load_q(it, it.v.n0 > 0 ? &p.tmqr : &p.tmq))) break;
        // step j of the item (j = 0..n) brings K(j) (for Q K of tile j) and
        // V(j-1) (for P V of tile j-1), the operands the issuer uses in the
        // same step, under one barrier
        for (int j = 0; j <= it.n_tiles; ++j) {
          const int gs = g + k + j, st = gs % kSt;
          if (!(ok = wait(&bar->step_empty[st], ((gs / kSt) & 1) ^ 1, abort, p.wait_ns))) break;
          // test hook: CTA 0 leaves its first step without copies or arrival, so
          // the issuer's wait for it is sure to run out
          if (p.drop_first_load && blockIdx.x == 0 && gs == 0) continue;
          uint64_t* full = &bar->step_full[st];
          mbar_arrive_expect_tx(full, (j < it.n_tiles ? kTile : 0) + (j > 0 ? kTile : 0));
          last_step[st] = gs;
          if (j < it.n_tiles) {
            const int kt = it.tile_at(j);
            uint8_t* dk = sK + st * kTile;
            for (int hh = 0; hh < kHalves; ++hh)
              tma_load_4d(dk + hh * kHalf, &p.tmk, full, 64 * hh, it.hk, kt * kBN, it.b, pol_kv);
          }
          if (j > 0) {
            const int kt = it.tile_at(j - 1);
            uint8_t* dv = sV + st * kTile;
            for (int hh = 0; hh < kHalves; ++hh)
              tma_load_4d(dv + hh * kHalf, &p.tmv, full, 64 * hh, it.hk, kt * kBN, it.b, pol_kv);
          }
          // the query at its own position for the visits after the renumbered ones
          if (j == it.v.n0 && j > 0 && j < it.n_tiles && !(ok = load_q(it, &p.tmq))) break;
        }
        g += it.n_tiles;
        ++k;
      }
    }
    __syncwarp();
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------- issuers
    // Issuer i issues head i's products.  Every mbarrier operation of an issuing
    // thread stalls it for hundreds of cycles while the tensor-core queue is only
    // a few products deep, so one thread alone leaves the pipe idle during its
    // waits.  Here each step is one group of products per head, and the groups
    // are issued strictly in turn (head 0's group t, head 1's group t, head 0's
    // group t + 1, ...): an issuer hands the turn on as soon as its group is
    // issued, and has done its own waits for the next group (operand tiles, its
    // head's P, O free) while the other's products were being issued.
    if (lane == 0) {
      const int i = warp - kMmaWarp;  // head of the pair
      // Descriptors are built once: moving a descriptor by `off` bytes adds
      // off / 16 to its start-address field (shared addresses stay below 256 KB,
      // so the 14-bit field never carries), which keeps the issue of the 16
      // products of a step off the critical path.
      const uint64_t dq = tc::sdesc_sw128(smem_u32(sQ + i * kTile), 16, 1024);
      const uint64_t dk = tc::sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv = tc::sdesc_sw128(smem_u32(sV), kHalf, 1024);
      // descriptors as 32-bit halves: only the low word (start address) moves,
      // and it never carries into the high word
      const uint32_t q_lo = (uint32_t)dq, q_hi = (uint32_t)(dq >> 32);
      const uint32_t k_lo = (uint32_t)dk, k_hi = (uint32_t)(dk >> 32);
      const uint32_t v_lo = (uint32_t)dv, v_hi = (uint32_t)(dv >> 32);
      auto mk = [](uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; };
      const uint32_t tS = tmem + i * 128, tO = tmem + 256 + i * 128;
      auto qk = [&](int sk) {
        const uint32_t b = k_lo + (uint32_t)((sk * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tS, mk(q_lo + off, q_hi), mk(b + off, k_hi), kIdescQK, kk > 0);
        }
        tc::commit(smem_u32(&bar->s_full[i]));
      };
      auto pv = [&](int sv, bool acc) {
        const uint32_t b = v_lo + (uint32_t)((sv * kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc::mma_bf16_ts(tO, tS + kk * 8, mk(b + ((kk * 2048) >> 4), v_hi), kIdescPV,
                          acc || kk > 0);
      };
      // t counts the groups this issuer has issued.  turn[0] completes a phase
      // each time issuer 1 hands over, turn[1] each time issuer 0 does; neither
      // can run two phases ahead of its waiter, since each hand-over needs the
      // other issuer's previous one.
      int g = 0, k = 0, kq = 0, t = 0;  // kq: Q loads consumed
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x) {
        const Item it = make_item(p, u);
        const int n = it.n_tiles, n0 = it.v.n0;
        if (n <= 0) continue;
        if (!(ok = wait(&bar->q_full, kq & 1, abort, p.wait_ns))) break;
        ++kq;
        for (int j = 0; j <= n; ++j, ++t) {
          const int gs = g + k + j, st = gs % kSt;  // step index: n + 1 steps per item
          // step gs brings K(j) for Q K of tile j and V(j-1) for P V of tile j-1
          if (!(ok = wait(&bar->step_full[st], (gs / kSt) & 1, abort, p.wait_ns))) break;
          // P_i(j-1) is written; the item's first P V overwrites O_i, which the
          // previous item's epilogue must have read out
          if (j > 0 && !(ok = wait(&bar->p_full[i], (g + j - 1) & 1, abort, p.wait_ns))) break;
          if (j == 1 && !(ok = wait(&bar->o_free[i], (k & 1) ^ 1, abort, p.wait_ns))) break;
          if (j < n && j == n0 && j > 0) {  // Reset PE: the second query has landed
            if (!(ok = wait(&bar->q_full, kq & 1, abort, p.wait_ns))) break;
            ++kq;
          }
          const bool turn = i == 0 ? (t == 0 || wait(&bar->turn[0], (t - 1) & 1, abort, p.wait_ns))
                                   : wait(&bar->turn[1], t & 1, abort, p.wait_ns);
          if (!(ok = turn)) break;
          tc::fence_after();
          if (j > 0) pv(st, j > 1);
          if (j < n)
            qk(st);
          else
            tc::commit(smem_u32(&bar->o_done[i]));
          tc::commit(smem_u32(&bar->step_empty[st]));
          // every Q K reading the current Q is issued: it may be replaced
          if (j == n - 1 || (j == n0 - 1 && n0 > 0)) tc::commit(smem_u32(&bar->q_empty));
          mbar_arrive(&bar->turn[i ^ 1]);
        }
        g += n;
        ++k;
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    const int i = warp >> 2;                 // head of the pair
    const int row = tid & 127;               // TMEM lane = query row in the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + i * 128 + lane_off, tO = tmem + 256 + i * 128 + lane_off;
    int g = 0, k = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x) {
      const Item it = make_item(p, u);
      if (it.n_tiles <= 0) continue;
      const int64_t qpos = it.q0 + row;
      // admitted key positions of this row: [0, min(P, qpos+1)) and [max(0, qpos-W+1), qpos]
      const int32_t a1 = keys_below(it.km, min((int64_t)it.P, qpos + 1));
      const int32_t b0 = keys_below(it.km, max((int64_t)0, qpos - p.W + 1));
      const int32_t b1 = keys_below(it.km, qpos + 1);
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_tiles; ++j) {
        // the tile's class and mask bounds are worked out before the wait, off
        // the S -> P critical path
        const int kt = it.tile_at(j);
        const int32_t ka = kt * kBN;
        const int32_t kb = min(it.km.n_keys, ka + kBN) - 1;
        const int mode = it.v.mode(j);
        const bool masked = tile_class(it.km, it.c0, it.q0r, it.q1r, ka, kb, it.P, p.W) != kFull ||
                            ka + kBN > it.km.n_keys || mode != kVisitAll;
        // kept columns: c < A1 (prefix keys) or B0 <= c < B1 (window keys); a
        // split tile's two visits keep only the keys before / after the prefix
        const int32_t A1 = mode == kVisitLaterPart ? 0 : a1 - ka;
        const int32_t B0 = mode == kVisitPrefixPart ? 0 : (mode == kVisitLaterPart ? max(b0, it.v.kP) : b0) - ka;
        const int32_t B1 = mode == kVisitPrefixPart ? 0 : b1 - ka;
        uint32_t km[kBN / 32];
        ok = wait(&bar->s_full[i], (g + j) & 1, abort, p.wait_ns);
        // tcgen05.ld / st are warp-collective (.sync.aligned): the warp decides
        // together and reconverges here after the per-thread spin
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc::fence_after();
        float alpha;
        if (masked) {
#pragma unroll
          for (int w = 0; w < kBN / 32; ++w) km[w] = keep_bits(32 * w, A1, B0, B1);
          alpha = softmax_tile<true>(tS, j, p.scale_log2, km, m_used, l);
        } else {
          alpha = softmax_tile<false>(tS, j, p.scale_log2, km, m_used, l);
        }
        if (__any_sync(0xffffffffu, alpha != 1.f)) {  // alpha is 1 on the other rows
          // O_i already holds every P V issued before S_i(j), which has completed,
          // and P_i(j) V is not issued before this thread arrives below
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::ld32(tO + c * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st32(tO + c * 32, o);
          }
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->p_full[i]);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      ok = wait(&bar->o_done[i], k & 1, abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const int32_t qrow = it.q0r + row;
      const float inv = 1.f / l;
      __nv_bfloat16* orow = p.out + (((int64_t)it.b * p.S + qrow) * p.hq + it.h0 + i) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld32(tO + c * 32, o);
        tc::wait_ld();
        if (c == D / 32 - 1) {  // O_i is read out: the next item may overwrite it
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar->o_free[i]);
        }
        if (qrow <= it.q1r) store_row_chunk(orow + c * 32, o, inv, p.out32 != 0);
      }
      if (qrow <= it.q1r)
        p.lse[((int64_t)it.b * p.hq + it.h0 + i) * p.S + qrow] =
            (m_used + __log2f(l)) * 0.69314718055994530942f;
      g += it.n_tiles;
      ++k;
    }
  }

  tc::fence_before();
  __syncthreads();
  if (*abort) {
    // A wait gave up.  Before shared and tensor memory are released, everything
    // issued must have landed: the producer waits (bounded) for each copy it
    // issued -- a completed phase answers at once, and no later phase of these
    // barriers can complete now -- and the issuer commits once more and waits
    // until all its products have completed.
    if (tid == 0) set_flag(p.status, PS_DEV_TIMEOUT);
    if (warp == kProducerWarp && lane == 0) {
      if (last_q >= 0) mbar_wait(&bar->q_full, (uint32_t)last_q, p.wait_ns);
#pragma unroll
      for (int s = 0; s < kSt; ++s)
        if (last_step[s] >= 0)
          mbar_wait(&bar->step_full[s], (uint32_t)((last_step[s] / kSt) & 1), p.wait_ns);
    } else if (warp >= kMmaWarp && lane == 0) {
      tc::commit(smem_u32(&bar->drain));
      mbar_wait(&bar->drain, 0, p.wait_ns);
    }
    __syncthreads();
  }
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, 512);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PrefillLayout {
  size_t q_off, k_off, v_off, qr_off, total;
  int32_t skv;
};

// [rotated Q][rotated K (ring rows, chunk)][gathered V, with a ring][Reset PE Q]
static PrefillLayout prefill_layout(int B, int S, int hq, int hkv, int D, int ring_rows,
                                    bool reset) {
  PrefillLayout L;
  L.skv = S + ring_rows;
  L.q_off = 0;
  L.k_off = align256((size_t)B * S * hq * D * 2);
  L.v_off = L.k_off + align256((size_t)B * L.skv * hkv * D * 2);
  L.qr_off = L.v_off + (ring_rows > 0 ? align256((size_t)B * L.skv * hkv * D * 2) : 0);
  L.total = L.qr_off + (reset ? align256((size_t)B * S * hq * D * 2) : 0);
  return L;
}

}  // namespace ps

using namespace ps;

// The tile kernel for head dim D: pairs of query heads when the group size is
// even, else one head per CTA.  cudaFuncSetAttribute is cheap and per device;
// it runs every time rather than behind a flag that would be wrong on a second
// device.
template <int D>
static ps_status_t launch_tiles(const PrefillParams& p, int group, int n_q_heads, int batch,
                                cudaStream_t s) {
  if (group % 2 == 0) {
    constexpr int smem = ws::smem_bytes<D>();
    if (cudaFuncSetAttribute(prefill_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return PS_ERR_CUDA;
    const int64_t n_items = (int64_t)p.nq * (n_q_heads / 2) * batch;
    if (n_items > 0x7fffffffLL) return PS_ERR_UNSUPPORTED;
    const int sms = device_sm_count();
    const int64_t grid = n_items < (sms > 0 ? sms : 148) ? n_items : (sms > 0 ? sms : 148);
    if (launch_dependent(prefill_pair_kernel<D>, dim3((unsigned)grid), dim3(ws::kThreads),
                         (size_t)smem, s, p) != cudaSuccess)
      return PS_ERR_CUDA;
  } else {
    constexpr int smem = Geom<D>::kSmemSingle;
    if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return PS_ERR_CUDA;
    dim3 grid((unsigned)p.nq, (unsigned)n_q_heads, (unsigned)batch);
    if (launch_dependent(prefill_kernel<D>, grid, dim3(128), (size_t)smem, s, p) != cudaSuccess)
      return PS_ERR_CUDA;
  }
  return PS_OK;
}

extern "C" ps_status_t ps_prefill_tile_grid(int32_t seqlen, int32_t q_start, int32_t prefix_len,
                                            int32_t window, int32_t with_ring, int32_t bm,
                                            int32_t bn, int32_t* nq, int32_t* nk) {
  if (!nq || !nk || seqlen < 1 || q_start < 0 || prefix_len < 0 || window < 1 || bm < 1 || bn < 1)
    return PS_ERR_INVALID_ARGUMENT;
  if ((int64_t)q_start + seqlen > 0x7fffffffLL) return PS_ERR_INVALID_ARGUMENT;
  const KeyMap m = make_keymap(seqlen, q_start, prefix_len, window, with_ring != 0);
  *nq = (seqlen + bm - 1) / bm;
  *nk = (m.n_keys + bn - 1) / bn;
  return PS_OK;
}

extern "C" ps_status_t ps_prefill_tile_classes(int32_t seqlen, int32_t q_start,
                                               int32_t prefix_len, int32_t window,
                                               int32_t with_ring, int32_t bm, int32_t bn,
                                               uint8_t* out, void* stream) {
  int32_t nq = 0, nk = 0;
  ps_status_t st = ps_prefill_tile_grid(seqlen, q_start, prefix_len, window, with_ring, bm, bn,
                                        &nq, &nk);
  if (st != PS_OK) return st;
  if (!out) return PS_ERR_INVALID_ARGUMENT;
  const KeyMap m = make_keymap(seqlen, q_start, prefix_len, window, with_ring != 0);
  const int64_t n = (int64_t)nq * nk;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  tile_classes_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      m, seqlen, q_start, prefix_len, window, bm, bn, nq, nk, out);
  return launch_status();
}

extern "C" ps_status_t ps_prefill_workspace_size(int32_t batch, int32_t seqlen, int32_t n_q_heads,
                                                 int32_t n_kv_heads, int32_t head_dim,
                                                 int32_t ring_rows_max, int32_t pe_mode,
                                                 size_t* bytes) {
  if (!bytes || batch < 1 || seqlen < 1 || n_q_heads < 1 || n_kv_heads < 1 || ring_rows_max < 0 ||
      n_q_heads % n_kv_heads || (pe_mode != PS_PE_CONTINUE && pe_mode != PS_PE_RESET))
    return PS_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return PS_ERR_UNSUPPORTED;
  *bytes = prefill_layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim, ring_rows_max,
                          pe_mode == PS_PE_RESET)
               .total;
  return PS_OK;
}

extern "C" ps_status_t ps_prefill(const void* q, const void* k, const void* v, int32_t batch,
                                  int32_t seqlen, const int32_t* q_start,
                                  const int32_t* prefix_len, int32_t window, int32_t n_q_heads,
                                  int32_t n_kv_heads, int32_t head_dim, float scale,
                                  double rope_theta, int32_t pe_mode, const ps_cache_desc* ring,
                                  const int32_t* ring_seq, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, int32_t* status, void* stream) {
  if (!q || !k || !v || !q_start || !prefix_len || !out || !lse) return PS_ERR_INVALID_ARGUMENT;
  if (batch < 1 || seqlen < 1 || window < 1 || n_q_heads < 1 || n_kv_heads < 1 ||
      n_q_heads % n_kv_heads || !(scale > 0.f) || !(rope_theta > 0.0))
    return PS_ERR_INVALID_ARGUMENT;
  if (pe_mode != PS_PE_CONTINUE && pe_mode != PS_PE_RESET) return PS_ERR_INVALID_ARGUMENT;
  if (ring && ring->pe_mode != pe_mode) return PS_ERR_INVALID_ARGUMENT;
  const bool reset = pe_mode == PS_PE_RESET;
  if (head_dim != 64 && head_dim != 128) return PS_ERR_UNSUPPORTED;
  if (batch > 65535 || n_q_heads > 65535) return PS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PS_ERR_ALIGNMENT;
  int ring_rows = 0;
  if (ring) {
    ps_status_t st = check_cache(ring);
    if (st != PS_OK) return st;
    if (ring->head_dim != head_dim || ring->n_kv_heads != n_kv_heads || ring->window != window)
      return PS_ERR_INVALID_ARGUMENT;
    ring_rows = ring->prefix_max + ring->window;
  }
  const PrefillLayout L =
      prefill_layout(batch, seqlen, n_q_heads, n_kv_heads, head_dim, ring_rows, reset);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PS_ERR_WORKSPACE;
  if (workspace_bytes < L.total) return PS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;

  GatherParams g;
  g.q = static_cast<const uint4*>(q);
  g.k = static_cast<const uint4*>(k);
  g.v = static_cast<const uint4*>(v);
  g.qh = reinterpret_cast<uint4*>(ws + L.q_off);
  g.qr = reset ? reinterpret_cast<uint4*>(ws + L.qr_off) : nullptr;
  g.kh = reinterpret_cast<uint4*>(ws + L.k_off);
  g.vg = ring ? reinterpret_cast<uint4*>(ws + L.v_off) : nullptr;
  g.q_start = q_start;
  g.prefix_len = prefix_len;
  g.status = status;
  g.k_pool = ring ? static_cast<const uint4*>(ring->k_pool) : nullptr;
  g.v_pool = ring ? static_cast<const uint4*>(ring->v_pool) : nullptr;
  g.ring_prefix = ring ? ring->prefix_len : nullptr;
  g.ring_seq = ring_seq;
  g.map = ring ? slot_map(ring) : SlotMap{};
  g.nseq = ring ? ring->nseq : 0;
  g.B = batch;
  g.S = seqlen;
  g.Skv = L.skv;
  g.hq = n_q_heads;
  g.hkv = n_kv_heads;
  g.W = window;
  make_rope_turns(rope_theta, head_dim, &g.turns);
  {
    const int64_t groups = ((int64_t)batch * seqlen + kRopeRows - 1) / kRopeRows;
    const int64_t extra = (int64_t)batch * (L.skv - seqlen) * n_kv_heads * (head_dim / 8);
    int64_t blocks = groups > (extra + 255) / 256 ? groups : (extra + 255) / 256;
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;  // 16 x 8 KB of smem per SM
    if (blocks > cap) blocks = cap;
    void (*pre)(GatherParams) =
        head_dim == 128 ? (reset ? rope_gather_kernel<true, 128> : rope_gather_kernel<false, 128>)
                        : (reset ? rope_gather_kernel<true, 64> : rope_gather_kernel<false, 64>);
    if (launch_dependent(pre, dim3((unsigned)blocks), dim3(256), 0, s, g) != cudaSuccess)
      return PS_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return PS_ERR_CUDA;
  }

  PrefillParams p;
  const uint64_t qd[4] = {(uint64_t)head_dim, (uint64_t)n_q_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t qs[3] = {(uint64_t)head_dim * 2, (uint64_t)n_q_heads * head_dim * 2,
                          (uint64_t)seqlen * n_q_heads * head_dim * 2};
  const uint64_t kd[4] = {(uint64_t)head_dim, (uint64_t)n_kv_heads, (uint64_t)L.skv, (uint64_t)batch};
  const uint64_t ks[3] = {(uint64_t)head_dim * 2, (uint64_t)n_kv_heads * head_dim * 2,
                          (uint64_t)L.skv * n_kv_heads * head_dim * 2};
  const uint64_t vd[4] = {(uint64_t)head_dim, (uint64_t)n_kv_heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t vs[3] = {(uint64_t)head_dim * 2, (uint64_t)n_kv_heads * head_dim * 2,
                          (uint64_t)seqlen * n_kv_heads * head_dim * 2};
  const uint32_t box[4] = {64u, 1u, (uint32_t)kBM, 1u};
  bool okm = encode_tmap(&p.tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ws + L.q_off, qd, qs, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_tmap(&p.tmqr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                         ws + (reset ? L.qr_off : L.q_off), qd, qs, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_tmap(&p.tmk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ws + L.k_off, kd, ks, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  if (ring)
    okm = okm && encode_tmap(&p.tmv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ws + L.v_off, kd, ks, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  else
    okm = okm && encode_tmap(&p.tmv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, vd, vs, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (!okm) return PS_ERR_CUDA;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  p.lse = lse;
  p.q_start = q_start;
  p.prefix_len = prefix_len;
  p.status = status;
  p.S = seqlen;
  p.hq = n_q_heads;
  p.hkv = n_kv_heads;
  p.W = window;
  p.with_ring = ring ? 1 : 0;
  p.reset = reset ? 1 : 0;
  const WaitHooks hooks = wait_hooks();
  p.wait_ns = hooks.wait_ns;
  p.drop_first_load = hooks.drop_first_load;
  p.nq = (seqlen + kBM - 1) / kBM;
  p.B = batch;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int group = n_q_heads / n_kv_heads;
  const ps_status_t st = head_dim == 128 ? launch_tiles<128>(p, group, n_q_heads, batch, s)
                                         : launch_tiles<64>(p, group, n_q_heads, batch, s);
  if (st != PS_OK) return st;
  return launch_status();
}
