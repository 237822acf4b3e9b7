// ps_decode.cu -- split-KV decode over the prefix and window slots, then an
// LSE-weighted combine.
//
// One generated token per sequence attends to its prefix and its last W
// positions, which after eviction are exactly ring slots [0, min(p+1, P+W))
// (njhaofan.com section "PrefixSliding如何丢掉中间Token？": once the window is
// full the per-step cost no longer grows; papers.ananclaw.com "伪代码" step
// decode).  The step is a memory-bound GEMV, so it runs on CUDA cores.
//
// Work split ("stream-K" over tiles): the (sequence, kv head) segments are laid
// end to end as 16-slot tiles, N tiles in all; warp w of the first NWe warps
// owns tiles [w*N/NWe, (w+1)*N/NWe), whatever the sequence lengths, where
// NWe = min(NW, ceil(N / kMinTilesPerWarp)): a short batch uses fewer warps, each
// with a few tiles in flight, rather than one tile on every warp of the grid and
// as many partial records to merge.  Each warp streams its
// tiles through a private STAGES-deep TMA ring in shared memory and writes
// one partial (unnormalised O, running max, running sum) per segment piece
// it touches.  Piece (warp w, segment sg) goes to record w + sg, which is
// unique because both indices only grow along the tile line; so NW + #segments
// records suffice.  The warps that take a segment's first and last tiles
// record themselves, and the combine kernel merges the records in between.
//
// Inside a warp, lane l holds D/32 consecutive elements of every row.  For a
// 16-row tile and two query heads the 32 partial dot products per lane are
// reduced by a butterfly transpose, after which lane l holds the score of row
// l % 16 for head l / 16; the softmax runs on those, and P V accumulates
// each lane's D/32 output elements of every head.  Eight warps per SM (two
// per scheduler) keep the scheduler busy while one warp waits on shared
// memory or shuffles.
#include "ps_internal.h"
#include "ps_rope.cuh"

namespace ps {

constexpr int kDecTile = 16;  // slots per tile
constexpr int kMinTilesPerWarp = 4;

// Warps that take tiles: all NW of the grid, or fewer for a short tile line.
__host__ __device__ __forceinline__ int64_t working_warps(int64_t N, int64_t NW) {
  const int64_t need = (N + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
  return need < NW ? need : NW;
}

struct DecodeParams {
  CUtensorMap tmk;  // 3D {D, Hkv, total_slots}, box {D, 1, kDecTile}
  CUtensorMap tmv;
  const __nv_bfloat16* q;  // [nseq, Hq, D]
  const __nv_bfloat16* k_new;  // [nseq, Hkv, D] raw K of the new tokens (fused append), or null
  const __nv_bfloat16* v_new;  // [nseq, Hkv, D]
  __nv_bfloat16* k_pool;       // the pools, written by the fused append
  __nv_bfloat16* v_pool;
  const int32_t* pos;
  const int32_t* prefix_len;
  int32_t* status;
  int32_t* seg_tiles;  // workspace: [nseq + 1] exclusive prefix of tiles per sequence
  int32_t* seg_warps;  // workspace: [nseq*Hkv][2] first and last warp of each segment
  float* rec;          // workspace: [NW + nseq*Hkv][rec_floats]
  SlotMap map;
  int32_t nseq, hq, hkv, window, prefix_max;
  int32_t nwarps_total;
  float scale_log2;  // softmax scale * log2(e)
  uint64_t wait_ns;  // bounded-wait limit
  int32_t drop_first_load;  // test hook: warp 0 of CTA 0 skips its first tile copy
  RopeTurns turns;
};

template <int D, int G>
struct DecShape {
  static constexpr int EPL = D / 32;                       // elements per lane
  static constexpr int TILE_BYTES = kDecTile * D * 2;      // one K or V tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int REC = ((G * D + 2 * G) + 3) & ~3;   // floats per record
  static constexpr int HP = G >= 2 ? 2 : 1;                // heads per score pass
  static constexpr int NPASS = G / HP;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Largest s in [0, nseq] with pfx[s] * hkv <= g (pfx non-decreasing, pfx[0] = 0).
__device__ __forceinline__ int find_seq(const int32_t* pfx, int nseq, int hkv, int64_t g) {
  int lo = 0, hi = nseq;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)pfx[mid] * hkv <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Position on the tile line: tile t of kv head h of sequence s (nt tiles per head).
struct TileIter {
  int64_t g;
  int s, h, t, nt;

  __device__ __forceinline__ void init(const int32_t* pfx, int nseq, int hkv, int64_t g0) {
    g = g0;
    s = find_seq(pfx, nseq, hkv, g0);
    nt = pfx[s + 1] - pfx[s];
    const int64_t r = g0 - (int64_t)pfx[s] * hkv;
    h = (int)(r / nt);
    t = (int)(r % nt);
  }
  __device__ __forceinline__ void next(const int32_t* pfx, int nseq, int hkv) {
    ++g;
    if (++t < nt) return;
    t = 0;
    if (++h < hkv) return;
    h = 0;
    do {
      ++s;
    } while (s < nseq && pfx[s + 1] == pfx[s]);  // sequences with no tiles own no line
    nt = s < nseq ? pfx[s + 1] - pfx[s] : 0;
  }
};

template <int EPL>
__device__ __forceinline__ void load_row_f32(const uint8_t* rowp, float (&x)[EPL]) {
  if constexpr (EPL == 4) {
    const uint2 w2 = *reinterpret_cast<const uint2*>(rowp);
    x[0] = bf16lo(w2.x); x[1] = bf16hi(w2.x); x[2] = bf16lo(w2.y); x[3] = bf16hi(w2.y);
  } else {
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(rowp);
    x[0] = bf16lo(w1); x[1] = bf16hi(w1);
  }
}

template <int D, int G, int WARPS, int STAGES, bool RESET>
__global__ void __launch_bounds__(WARPS * 32, 1)
    decode_partial_kernel(const __grid_constant__ DecodeParams p) {
  using S = DecShape<D, G>;
  constexpr int EPL = S::EPL, HP = S::HP, NPASS = S::NPASS, TS = kDecTile;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + WARPS * STAGES * S::STAGE_BYTES);
  float* pbuf_all = reinterpret_cast<float*>(bars + WARPS * STAGES);  // [WARPS][G * TS]
  int32_t* pfx = reinterpret_cast<int32_t*>(pbuf_all + WARPS * G * TS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[warp * STAGES + st], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmk);
    prefetch_tmap(&p.tmv);
  }
  grid_dependency_wait();  // the appended tokens and the workspace come from earlier work
  allow_dependents();

  // 1) tiles per sequence and their exclusive prefix (warp 0, 32 sequences at a time)
  if (warp == 0) {
    int32_t run = 0;
    for (int b0 = 0; b0 < p.nseq; b0 += 32) {
      const int s = b0 + lane;
      int32_t n = 0;
      if (s < p.nseq) {
        const int32_t P = p.prefix_len[s], ps_ = p.pos[s];
        int32_t bad = 0;
        if (P < 0 || P > p.prefix_max) bad |= PS_DEV_BAD_PREFIX;
        if (ps_ < 0) bad |= PS_DEV_BAD_POS;
        if (!p.map.seq_ok(s)) bad |= PS_DEV_BAD_SLOT;
        if (bad) {
          if (blockIdx.x == 0) set_flag(p.status, bad);
        } else {
          const int64_t L = min((int64_t)ps_ + 1, (int64_t)P + p.window);
          n = (int32_t)((L + TS - 1) / TS);
        }
      }
      int32_t x = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (s < p.nseq) pfx[s] = run + x - n;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) pfx[p.nseq] = run;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= p.nseq; i += blockDim.x) p.seg_tiles[i] = pfx[i];

  const int64_t N = (int64_t)pfx[p.nseq] * p.hkv;
  const int64_t NWe = working_warps(N, p.nwarps_total);
  const int w = blockIdx.x * WARPS + warp;
  if (w >= NWe) return;  // no block-wide barrier follows
  const int64_t lo = N * w / NWe, hi = N * (w + 1) / NWe;  // never empty: N >= NWe

  uint8_t* my_tiles = tiles + warp * STAGES * S::STAGE_BYTES;
  uint64_t* my_bars = bars + warp * STAGES;
  float* pbuf = pbuf_all + warp * G * TS;

  const uint64_t pol = policy_evict_first();
  TileIter nxt;  // next tile to request (lane 0 only)
  auto issue = [&](int st) {
    int64_t r = p.map.row(nxt.s, nxt.t * TS);  // a tile never straddles a block
    if (r < 0) {  // block outside the pool: flag it and read block 0 instead
      set_flag(p.status, PS_DEV_BAD_SLOT);
      r = 0;
    }
    const int32_t row0 = (int32_t)r;
    uint64_t* bar = &my_bars[st];
    uint8_t* dst = my_tiles + st * S::STAGE_BYTES;
    mbar_arrive_expect_tx(bar, S::STAGE_BYTES);
    tma_load_3d(dst, &p.tmk, bar, 0, nxt.h, row0, pol);
    tma_load_3d(dst + S::TILE_BYTES, &p.tmv, bar, 0, nxt.h, row0, pol);
  };
  if (lane == 0) {
    nxt.init(pfx, p.nseq, p.hkv, lo);
    for (int k = 0; k < STAGES && nxt.g < hi; ++k) {
      // test hook: no copy and no arrival, so the first wait is sure to run out
      if (!(k == 0 && p.drop_first_load && blockIdx.x == 0 && warp == 0)) issue(k);
      nxt.next(pfx, p.nseq, p.hkv);
    }
  }

  TileIter cur;
  cur.init(pfx, p.nseq, p.hkv, lo);
  uint32_t parity = 0;  // bit st = parity expected next on stage st
  float qf[G][EPL], qr[G][EPL], acc[G][EPL], m[NPASS], lsum[NPASS];
  int cur_L = 0;
  int cur_slot = -1;      // fused append: the new token's slot in the current sequence
  float kc[EPL], ksn[EPL];  // fused append: (cos, sin) of this lane's pairs at pos[s]
  int32_t seg_P = 0;      // prefix length of the current sequence
  bool seg_reset = false; // Reset PE changes this sequence's prefix scores
  bool ok = true;
  int64_t consumed = lo;
  int st = 0;

  for (; cur.g < hi; cur.next(pfx, p.nseq, p.hkv)) {
    const int s = cur.s, h = cur.h, t = cur.t;
    if (lane == 0) {  // segment ends: the combine reads its warps from here
      if (t == 0) p.seg_warps[2 * ((int64_t)s * p.hkv + h)] = w;
      if (t == cur.nt - 1) p.seg_warps[2 * ((int64_t)s * p.hkv + h) + 1] = w;
    }
    if (cur.g == lo || t == 0) {
      // new segment piece: rotate the group's queries at position pos[s]
      const int32_t ppos = p.pos[s];
      seg_P = p.prefix_len[s];
      cur_L = (int)min((int64_t)ppos + 1, (int64_t)seg_P + p.window);
      // Reset PE renumbers the cache 0..L-1 and the query as L-1: window keys
      // keep their distance to the query, prefix keys see it rotated at L-1
      const int32_t rpos = cur_L - 1;
      seg_reset = RESET && rpos != ppos;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const __nv_bfloat16* qrow = p.q + ((int64_t)s * p.hq + h * G + gg) * D + lane * EPL;
        float x[EPL];
        load_row_f32<EPL>(reinterpret_cast<const uint8_t*>(qrow), x);
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          // half-split RoPE: element i pairs with i + D/2, held by lane ^ 16
          const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
          const int i = (lane & 15) * EPL + e;
          float c, sn;
          rope_cos_sin(ppos, p.turns.f[i], c, sn);
          kc[e] = c;
          ksn[e] = sn;
          const float y = (lane < 16) ? (x[e] * c - partner * sn) : (x[e] * c + partner * sn);
          // rotated Q is rounded to bf16, as the cache stores rotated K
          qf[gg][e] = __bfloat162float(__float2bfloat16_rn(y)) * p.scale_log2;
          qr[gg][e] = qf[gg][e];
          if (RESET && seg_reset) {
            rope_cos_sin(rpos, p.turns.f[i], c, sn);
            const float yr = (lane < 16) ? (x[e] * c - partner * sn) : (x[e] * c + partner * sn);
            qr[gg][e] = __bfloat162float(__float2bfloat16_rn(yr)) * p.scale_log2;
          }
          acc[gg][e] = 0.f;
        }
      }
#pragma unroll
      for (int ps_ = 0; ps_ < NPASS; ++ps_) {
        m[ps_] = -INFINITY;
        lsum[ps_] = 0.f;
      }
      cur_slot = p.k_new ? ring_slot(ppos, seg_P, p.window) : -1;
    }

    // the lanes decide together: shuffles and the drain below need the whole warp
    if (!__all_sync(0xffffffffu, mbar_wait(&my_bars[st], (parity >> st) & 1u, p.wait_ns))) {
      ok = false;
      break;
    }
    parity ^= 1u << st;
    consumed = cur.g + 1;

    // Fused append (ps_decode_append): the tile holding the new token's slot
    // came with the slot's previous occupant.  Put the new token's K (rotated
    // at pos[s] exactly as ps_kv_append does) and V in its place, in the tile
    // and in the pool; this warp is the only reader of this head's part of
    // that row in this launch.
    if (cur_slot >= 0 && t == cur_slot / TS) {
      const int64_t src = ((int64_t)s * p.hkv + h) * D + lane * EPL;
      float x[EPL];
      load_row_f32<EPL>(reinterpret_cast<const uint8_t*>(p.k_new + src), x);
      float rk[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
        rk[e] = lane < 16 ? rope_first(x[e], partner, kc[e], ksn[e])
                          : rope_second(partner, x[e], kc[e], ksn[e]);
      }
      uint32_t kw[EPL / 2], vw[EPL / 2];
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        kw[e] = pack_bf16(rk[2 * e], rk[2 * e + 1]);
        vw[e] = reinterpret_cast<const uint32_t*>(p.v_new + src)[e];
      }
      uint8_t* ks = my_tiles + st * S::STAGE_BYTES + (cur_slot % TS) * (D * 2) + lane * (EPL * 2);
      const int64_t row = p.map.row(s, cur_slot);
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        reinterpret_cast<uint32_t*>(ks)[e] = kw[e];
        reinterpret_cast<uint32_t*>(ks + S::TILE_BYTES)[e] = vw[e];
      }
      if (row >= 0) {
        const int64_t dst = (row * p.hkv + h) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL / 2; ++e) {
          reinterpret_cast<uint32_t*>(p.k_pool + dst)[e] = kw[e];
          reinterpret_cast<uint32_t*>(p.v_pool + dst)[e] = vw[e];
        }
      }
      __syncwarp();
    }

    const uint8_t* kt = my_tiles + st * S::STAGE_BYTES;
    const uint8_t* vt = kt + S::TILE_BYTES;
    const int nvalid = min(TS, cur_L - t * TS);
    const int myrow = lane & (TS - 1);

    // ---- scores of pass ps_: 16 rows x HP heads of partial dot products per
    // lane, reduced so that lane l holds row l % 16 of head ps_ * HP + l / 16
    // rows j < npre (the Reset PE prefix rows of the tile) use qr, the rest qf
    auto tile_scores = [&](int npre, int ps_) -> float {
      float v[32];
#pragma unroll
      for (int j = 0; j < TS; ++j) {
        float k4[EPL];
        load_row_f32<EPL>(kt + j * (D * 2) + lane * (EPL * 2), k4);
        const bool r = j < npre;
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
          const float(&qq)[EPL] = r ? qr[ps_ * HP + hh] : qf[ps_ * HP + hh];
          float a = qq[0] * k4[0];
#pragma unroll
          for (int e = 1; e < EPL; ++e) a = fmaf(qq[e], k4[e], a);
          v[hh * TS + j] = a;
        }
      }
      if constexpr (HP == 1) {  // one head: fold the two lane halves, then transpose
#pragma unroll
        for (int i = 0; i < TS; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 16);
      } else {
        // butterfly transpose-reduce: after the step at offset o a lane keeps
        // the half of its partials whose index has bit o equal to its lane bit
        const bool up = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float send = up ? v[i] : v[i + 16];
          const float keep = up ? v[i + 16] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = up ? v[i] : v[i + o];
          const float keep = up ? v[i + o] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      return v[0];
    };

#pragma unroll
    for (int ps_ = 0; ps_ < NPASS; ++ps_) {
      // Reset PE: the tile's first npre rows are prefix slots (uniform per tile)
      const int npre = RESET && seg_reset ? min(TS, max(0, seg_P - t * TS)) : 0;
      const float sc = (!RESET || npre == 0) ? tile_scores(0, ps_) : tile_scores(npre, ps_);
      // lane l: score of row l % 16 for head ps_ * HP + l / 16 (log2 domain)
      const float x = myrow < nvalid ? sc : -INFINITY;
      float tmax = x;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float mn = fmaxf(m[ps_], tmax);
      const float alpha = fast_exp2(m[ps_] - mn);
      const float pr = fast_exp2(x - mn);
      lsum[ps_] = lsum[ps_] * alpha + pr;
      m[ps_] = mn;
      if (HP == 2 || lane < 16) pbuf[ps_ * 32 + lane] = pr;
#pragma unroll
      for (int hh = 0; hh < HP; ++hh) {
        const float a_h = __shfl_sync(0xffffffffu, alpha, hh * 16);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[ps_ * HP + hh][e] *= a_h;
      }
    }
    __syncwarp();

    // ---- O += P V over the valid rows (invalid rows may hold stale values)
    auto pv_row = [&](int j) {
      float v4[EPL];
      load_row_f32<EPL>(vt + j * (D * 2) + lane * (EPL * 2), v4);
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float pj = pbuf[gg * TS + j];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[gg][e] = fmaf(pj, v4[e], acc[gg][e]);
      }
    };
    if (nvalid == TS) {
#pragma unroll
      for (int j = 0; j < TS; ++j) pv_row(j);
    } else {
      for (int j = 0; j < nvalid; ++j) pv_row(j);
    }

    // ---- end of this warp's piece of the segment: write the partial record
    if (t == cur.nt - 1 || cur.g == hi - 1) {
      float* rec = p.rec + (size_t)(w + (int64_t)s * p.hkv + h) * S::REC;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float* o = rec + gg * D + lane * EPL;
        if constexpr (EPL == 4) {
          *reinterpret_cast<float4*>(o) = make_float4(acc[gg][0], acc[gg][1], acc[gg][2], acc[gg][3]);
        } else {
          *reinterpret_cast<float2*>(o) = make_float2(acc[gg][0], acc[gg][1]);
        }
      }
#pragma unroll
      for (int ps_ = 0; ps_ < NPASS; ++ps_) {
        float tot = lsum[ps_];
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if ((lane & 15) == 0 && (HP == 2 || lane == 0)) {
          const int gg = ps_ * HP + (lane >> 4);
          rec[G * D + gg] = m[ps_];
          rec[G * D + G + gg] = tot;
        }
      }
    }
    __syncwarp();
    if (lane == 0 && nxt.g < hi) {
      fence_proxy_async_smem();
      issue(st);
      nxt.next(pfx, p.nseq, p.hkv);
    }
    st = st + 1 == STAGES ? 0 : st + 1;
  }

  if (!ok) {
    // a wait gave up: report, then let the copies already issued land (bounded)
    if (lane == 0) set_flag(p.status, PS_DEV_TIMEOUT);
    const int64_t issued_end = min(hi, consumed + STAGES);
    for (int64_t g = consumed + 1; g < issued_end; ++g) {
      const int sg = (int)((g - lo) % STAGES);
      if (!mbar_wait(&my_bars[sg], (parity >> sg) & 1u, p.wait_ns)) break;
      parity ^= 1u << sg;
    }
  }
}

struct CombineParams {
  const float* rec;
  const int32_t* seg_tiles;
  const int32_t* seg_warps;
  __nv_bfloat16* out;  // [nseq, Hq, D]
  float* lse;          // [nseq, Hq]
  int32_t nseq, hq, hkv, nwarps_total;
};

// One CTA of eight warps per (sequence, query head): merge the partial softmax
// records of the warps that covered its segment, its first through last warp
// as the partial kernel recorded them (every working warp owns at least one
// tile, so each of them wrote a record).  The warps take an eighth of the
// records each, read them eight at a time (loads first, then the
// running-maximum merges), and merge their results through shared memory, so a
// segment spread over many warps (a short batch) costs a few load latencies,
// not one per record.
constexpr int kCombineWarps = 8;

template <int D, int G>
__global__ void __launch_bounds__(kCombineWarps * 32)
    decode_combine_kernel(const __grid_constant__ CombineParams p) {
  using S = DecShape<D, G>;
  constexpr int EPL = S::EPL, NWARP = kCombineWarps, U = 8;
  __shared__ float sm_m[NWARP], sm_l[NWARP];
  __shared__ float sm_a[NWARP][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();  // the partial records come from the previous kernel
  allow_dependents();
  const int64_t gw = blockIdx.x;  // (sequence, query head)
  if (gw >= (int64_t)p.nseq * p.hq) return;
  const int s = (int)(gw / p.hq), hq = (int)(gw % p.hq);
  const int h = hq / G, gg = hq % G;
  const int32_t nt = p.seg_tiles[s + 1] - p.seg_tiles[s];
  __nv_bfloat16* o = p.out + gw * D + lane * EPL;
  if (nt == 0) {  // sequence rejected by the device checks
    if (warp == 0) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[e] = __float2bfloat16_rn(0.f);
      if (lane == 0) p.lse[gw] = -INFINITY;
    }
    return;
  }
  const int64_t sg = (int64_t)s * p.hkv + h;
  const int w0 = p.seg_warps[2 * sg];
  const int R = p.seg_warps[2 * sg + 1] - w0 + 1;
  const int k_lo = R * warp / NWARP, k_hi = R * (warp + 1) / NWARP;
  float M = -INFINITY, l = 0.f, a[EPL] = {};
  for (int k0 = k_lo; k0 < k_hi; k0 += U) {
    float mw[U], lw[U], aw[U][EPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float* r = p.rec + (size_t)(w0 + min(k0 + u, k_hi - 1) + sg) * S::REC;
      mw[u] = r[G * D + gg];
      lw[u] = r[G * D + G + gg];
#pragma unroll
      for (int e = 0; e < EPL; ++e) aw[u][e] = r[gg * D + lane * EPL + e];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (k0 + u >= k_hi) break;
      const float mn = fmaxf(M, mw[u]);
      const float f_old = fast_exp2(M - mn), f_new = fast_exp2(mw[u] - mn);
      l = l * f_old + lw[u] * f_new;
#pragma unroll
      for (int e = 0; e < EPL; ++e) a[e] = a[e] * f_old + aw[u][e] * f_new;
      M = mn;
    }
  }
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) sm_a[warp][lane * EPL + e] = a[e];
  __syncthreads();
  if (warp != 0) return;
  float Mt = sm_m[0];
#pragma unroll
  for (int x = 1; x < NWARP; ++x) Mt = fmaxf(Mt, sm_m[x]);
  float lt = 0.f, at[EPL] = {};
#pragma unroll
  for (int x = 0; x < NWARP; ++x) {
    if (sm_m[x] == -INFINITY) continue;  // a warp with no records
    const float f = fast_exp2(sm_m[x] - Mt);
    lt += sm_l[x] * f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) at[e] += sm_a[x][lane * EPL + e] * f;
  }
  const float inv = 1.f / lt;
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = __float2bfloat16_rn(at[e] * inv);
  if (lane == 0) p.lse[gw] = (Mt + log2f(lt)) * 0.69314718055994530942f;
}

// ----------------------------------------------------------------- host ----
constexpr int kDecWarps = 8;
constexpr int kDecStages = 3;

template <int D, int G>
static size_t dec_smem_bytes(int nseq) {
  using S = DecShape<D, G>;
  return (size_t)kDecWarps * kDecStages * S::STAGE_BYTES + kDecWarps * kDecStages * 8 +
         kDecWarps * G * kDecTile * 4 + (size_t)(nseq + 1) * 4;
}

struct DecPlan {
  int grid = 0, nwarps = 0;
  size_t smem = 0, rec_floats = 0;
  void (*partial)(DecodeParams) = nullptr;
  void (*combine)(CombineParams) = nullptr;
};

// The grid (hence the workspace size) is the same for both position-encoding
// variants: it uses the smaller of their occupancies.
template <int D, int G>
static bool plan_for(int nseq, bool reset, DecPlan* pl) {
  auto kc = decode_partial_kernel<D, G, kDecWarps, kDecStages, false>;
  auto kr = decode_partial_kernel<D, G, kDecWarps, kDecStages, true>;
  pl->smem = dec_smem_bytes<D, G>(nseq);
  if (pl->smem > 227 * 1024) return false;
  int per_sm = 0, per_sm_r = 0;
  if (cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl->smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl->smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kc, kDecWarps * 32, pl->smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_r, kr, kDecWarps * 32, pl->smem) !=
          cudaSuccess)
    return false;
  per_sm = per_sm < per_sm_r ? per_sm : per_sm_r;
  if (per_sm < 1) return false;
  auto kp = reset ? kr : kc;
  const int sms = device_sm_count();
  if (sms < 1) return false;
  pl->grid = sms * per_sm;
  pl->nwarps = pl->grid * kDecWarps;
  pl->rec_floats = DecShape<D, G>::REC;
  pl->partial = reinterpret_cast<void (*)(DecodeParams)>(kp);
  pl->combine = reinterpret_cast<void (*)(CombineParams)>(decode_combine_kernel<D, G>);
  return true;
}

static bool make_plan(int D, int G, int nseq, bool reset, DecPlan* pl) {
#define PS_DEC_CASE(DD, GG) \
  if (D == DD && G == GG) return plan_for<DD, GG>(nseq, reset, pl);
  PS_DEC_CASE(128, 1) PS_DEC_CASE(128, 2) PS_DEC_CASE(128, 4) PS_DEC_CASE(128, 8)
  PS_DEC_CASE(64, 1) PS_DEC_CASE(64, 2) PS_DEC_CASE(64, 4) PS_DEC_CASE(64, 8)
#undef PS_DEC_CASE
  return false;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static size_t dec_ws_bytes(const DecPlan& pl, int nseq, int hkv) {
  return align256((size_t)(nseq + 1) * 4) + align256((size_t)nseq * hkv * 2 * 4) +
         (size_t)(pl.nwarps + (size_t)nseq * hkv) * pl.rec_floats * 4;
}

static ps_status_t check_heads(int hq, int hkv, int D) {
  if (hq < 1 || hkv < 1 || hq % hkv) return PS_ERR_INVALID_ARGUMENT;
  const int G = hq / hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PS_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PS_ERR_UNSUPPORTED;
  return PS_OK;
}

}  // namespace ps

using namespace ps;

static constexpr int kMaxDecodeSeqs = 4096;

extern "C" ps_status_t ps_decode_workspace_size(int32_t nseq, int32_t n_q_heads, int32_t n_kv_heads,
                                                int32_t head_dim, size_t* bytes) {
  if (!bytes || nseq < 1) return PS_ERR_INVALID_ARGUMENT;
  if (nseq > kMaxDecodeSeqs) return PS_ERR_UNSUPPORTED;
  ps_status_t st = check_heads(n_q_heads, n_kv_heads, head_dim);
  if (st != PS_OK) return st;
  DecPlan pl;
  if (!make_plan(head_dim, n_q_heads / n_kv_heads, nseq, false, &pl)) return PS_ERR_CUDA;
  *bytes = dec_ws_bytes(pl, nseq, n_kv_heads);
  return PS_OK;
}

// Validates the decode arguments and fills the launch parameters of both kernels.
static ps_status_t prepare_decode(const ps_cache_desc* cache, int32_t n_q_heads, const void* ws,
                                  size_t ws_bytes, DecPlan* pl) {
  ps_status_t st = check_cache(cache);
  if (st != PS_OK) return st;
  st = check_heads(n_q_heads, cache->n_kv_heads, cache->head_dim);
  if (st != PS_OK) return st;
  if (cache->nseq > kMaxDecodeSeqs) return PS_ERR_UNSUPPORTED;
  if (!make_plan(cache->head_dim, n_q_heads / cache->n_kv_heads, cache->nseq,
                 cache->pe_mode == PS_PE_RESET, pl))
    return PS_ERR_CUDA;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return PS_ERR_WORKSPACE;
  if (ws_bytes < dec_ws_bytes(*pl, cache->nseq, cache->n_kv_heads)) return PS_ERR_WORKSPACE;
  return PS_OK;
}

static int32_t* seg_warps_of(void* ws, int nseq) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + align256((size_t)(nseq + 1) * 4));
}

static float* records_of(void* ws, int nseq, int hkv) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256((size_t)(nseq + 1) * 4) +
                                  align256((size_t)nseq * hkv * 2 * 4));
}

// The partial launch, with (k_new, v_new) the fused append's new tokens or null.
static ps_status_t decode_partial(const ps_cache_desc* cache, const void* q, const void* k_new,
                                  const void* v_new, const int32_t* pos, int32_t n_q_heads,
                                  float scale, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (!q || !pos || !(scale > 0.f)) return PS_ERR_INVALID_ARGUMENT;
  DecPlan pl;
  ps_status_t st = prepare_decode(cache, n_q_heads, workspace, workspace_bytes, &pl);
  if (st != PS_OK) return st;
  if (!aligned16(q)) return PS_ERR_ALIGNMENT;
  if ((k_new || v_new) && (!k_new || !v_new)) return PS_ERR_INVALID_ARGUMENT;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PS_ERR_ALIGNMENT;
  const int D = cache->head_dim, hkv = cache->n_kv_heads, nseq = cache->nseq;
  DecodeParams p;
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)hkv, (uint64_t)cache->total_slots};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)hkv * D * 2};
  const uint32_t box[3] = {(uint32_t)D, 1u, (uint32_t)kDecTile};
  if (!encode_tmap(&p.tmk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, cache->k_pool, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap(&p.tmv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, cache->v_pool, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return PS_ERR_CUDA;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.k_pool = static_cast<__nv_bfloat16*>(cache->k_pool);
  p.v_pool = static_cast<__nv_bfloat16*>(cache->v_pool);
  p.pos = pos;
  p.prefix_len = cache->prefix_len;
  p.status = cache->status;
  p.seg_tiles = static_cast<int32_t*>(workspace);
  p.seg_warps = seg_warps_of(workspace, nseq);
  p.rec = records_of(workspace, nseq, hkv);
  p.map = slot_map(cache);
  p.nseq = nseq;
  p.hq = n_q_heads;
  p.hkv = hkv;
  p.window = cache->window;
  p.prefix_max = cache->prefix_max;
  p.nwarps_total = pl.nwarps;
  p.scale_log2 = scale * 1.4426950408889634f;
  const WaitHooks hooks = wait_hooks();
  p.wait_ns = hooks.wait_ns;
  p.drop_first_load = hooks.drop_first_load;
  make_rope_turns(cache->rope_theta, D, &p.turns);
  if (launch_dependent(pl.partial, dim3(pl.grid), dim3(kDecWarps * 32), pl.smem,
                       (cudaStream_t)stream, p) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}

extern "C" ps_status_t ps_decode_partial(const ps_cache_desc* cache, const void* q,
                                         const int32_t* pos, int32_t n_q_heads, float scale,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  return decode_partial(cache, q, nullptr, nullptr, pos, n_q_heads, scale, workspace,
                        workspace_bytes, stream);
}

extern "C" ps_status_t ps_decode_combine(const ps_cache_desc* cache, int32_t n_q_heads, void* out,
                                         float* lse, const void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (!out || !lse) return PS_ERR_INVALID_ARGUMENT;
  DecPlan pl;
  ps_status_t st = prepare_decode(cache, n_q_heads, workspace, workspace_bytes, &pl);
  if (st != PS_OK) return st;
  if (!aligned16(out)) return PS_ERR_ALIGNMENT;
  const int nseq = cache->nseq;
  CombineParams c;
  c.rec = records_of(const_cast<void*>(workspace), nseq, cache->n_kv_heads);
  c.seg_tiles = static_cast<const int32_t*>(workspace);
  c.seg_warps = seg_warps_of(const_cast<void*>(workspace), nseq);
  c.out = static_cast<__nv_bfloat16*>(out);
  c.lse = lse;
  c.nseq = nseq;
  c.hq = n_q_heads;
  c.hkv = cache->n_kv_heads;
  c.nwarps_total = pl.nwarps;
  const int64_t warps = (int64_t)nseq * n_q_heads;
  if (launch_dependent(pl.combine, dim3((unsigned)warps), dim3(kCombineWarps * 32), 0,
                       (cudaStream_t)stream, c) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}

extern "C" ps_status_t ps_decode(const ps_cache_desc* cache, const void* q, const int32_t* pos,
                                 int32_t n_q_heads, float scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!out || !lse) return PS_ERR_INVALID_ARGUMENT;
  ps_status_t st = ps_decode_partial(cache, q, pos, n_q_heads, scale, workspace, workspace_bytes,
                                     stream);
  if (st != PS_OK) return st;
  return ps_decode_combine(cache, n_q_heads, out, lse, workspace, workspace_bytes, stream);
}

extern "C" ps_status_t ps_decode_append(const ps_cache_desc* cache, const void* q, const void* k,
                                        const void* v, const int32_t* pos, int32_t n_q_heads,
                                        float scale, void* out, float* lse, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!out || !lse || !k || !v) return PS_ERR_INVALID_ARGUMENT;
  ps_status_t st = decode_partial(cache, q, k, v, pos, n_q_heads, scale, workspace,
                                  workspace_bytes, stream);
  if (st != PS_OK) return st;
  return ps_decode_combine(cache, n_q_heads, out, lse, workspace, workspace_bytes, stream);
}
