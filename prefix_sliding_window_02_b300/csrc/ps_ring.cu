// ps_ring.cu -- ring-slot mapping and the RoPE + append kernel.
//
// The cache keeps P fixed prefix slots and W rotating window slots per
// sequence (njhaofan.com section "PrefixSliding如何丢掉中间Token？"; the
// "伪代码" section of the papers.ananclaw.com explainer fixes the cache size at
// prefix_len + W).  Keys are rotated once, at their absolute position, when
// they are appended, and never again (Continue PE, agihunt.info paragraph on
// position encodings).
#include "ps_internal.h"

namespace ps {

__global__ void ring_slots_kernel(const int32_t* __restrict__ pos, const int32_t* __restrict__ P,
                                  int32_t W, int32_t* __restrict__ slot, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int32_t p = pos[i], pp = P[i];
    slot[i] = (p < 0 || pp < 0) ? -1 : ring_slot(p, pp, W);
  }
}

struct AppendParams {
  const uint4* k;  // [T, Hkv, D] bf16 as 16-byte vectors
  const uint4* v;
  uint4* kp;       // [total_slots, Hkv, D]
  uint4* vp;
  const int32_t* seq_idx;
  const int32_t* pos0;
  const int32_t* cu;
  const int64_t* slot_base;
  const int32_t* prefix_len;
  int32_t* status;
  int64_t n_tokens;
  int64_t total_slots;
  int32_t nrun, nseq, hkv, head_dim, window, capacity, prefix_max;
  RopeTurns turns;
};

// One thread per (token, kv head, group of 8 rotation pairs): it loads the 8
// elements of the first half and their 8 partners in the second half (two
// 16-byte loads), rotates them in fp32 and stores bf16 (round to nearest even).
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
  const int groups = p.head_dim / 16;
  const int vec_per_row = p.head_dim / 8;  // 16-byte vectors per head row
  const int64_t items = p.n_tokens * p.hkv * groups;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(it % groups);
    const int64_t rest = it / groups;
    const int h = (int)(rest % p.hkv);
    const int64_t t = rest / p.hkv;
    // run r: the largest r with cu[r] <= t
    int lo = 0, hi = p.nrun - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (p.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int64_t c0 = p.cu[lo], c1 = p.cu[lo + 1];
    if (!(c0 <= t && t < c1)) { set_flag(p.status, PS_DEV_BAD_RUN); continue; }
    const int32_t s = p.seq_idx[lo];
    if (s < 0 || s >= p.nseq) { set_flag(p.status, PS_DEV_BAD_SEQ); continue; }
    const int32_t P = p.prefix_len[s];
    if (P < 0 || P > p.prefix_max) { set_flag(p.status, PS_DEV_BAD_PREFIX); continue; }
    const int64_t base = p.slot_base[s];
    if (base < 0 || base + p.capacity > p.total_slots) { set_flag(p.status, PS_DEV_BAD_SLOT); continue; }
    const int64_t first = p.pos0[lo];
    const int64_t last = first + (c1 - c0) - 1;
    if (first < 0 || last > 0x7fffffffLL) { set_flag(p.status, PS_DEV_BAD_POS); continue; }
    const int32_t pos = (int32_t)(first + (t - c0));
    // A window position is overwritten later in the same run once a position
    // W further on is also in it: only prefix positions and the last W survive.
    if (!(pos < P || (int64_t)pos > last - p.window)) continue;
    const int64_t row = base + ring_slot(pos, P, p.window);

    const int64_t src = (t * p.hkv + h) * vec_per_row;
    const int64_t dst = (row * p.hkv + h) * vec_per_row;
    const int half_vec = vec_per_row / 2;
    uint4 a = p.k[src + g], b = p.k[src + half_vec + g];
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
    const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b);
    uint4 ra, rb;
    uint32_t* raw = reinterpret_cast<uint32_t*>(&ra);
    uint32_t* rbw = reinterpret_cast<uint32_t*>(&rb);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float c0f, s0f, c1f, s1f;
      rope_cos_sin(pos, p.turns.f[8 * g + 2 * e], c0f, s0f);
      rope_cos_sin(pos, p.turns.f[8 * g + 2 * e + 1], c1f, s1f);
      const float x0 = bf16lo(aw[e]), x1 = bf16hi(aw[e]);  // first-half elements
      const float y0 = bf16lo(bw[e]), y1 = bf16hi(bw[e]);  // their partners
      raw[e] = pack_bf16(x0 * c0f - y0 * s0f, x1 * c1f - y1 * s1f);
      rbw[e] = pack_bf16(y0 * c0f + x0 * s0f, y1 * c1f + x1 * s1f);
    }
    p.kp[dst + g] = ra;
    p.kp[dst + half_vec + g] = rb;
    p.vp[dst + g] = p.v[src + g];
    p.vp[dst + half_vec + g] = p.v[src + half_vec + g];
  }
}

}  // namespace ps

using namespace ps;

extern "C" ps_status_t ps_ring_slots(const int32_t* pos, const int32_t* prefix_len, int32_t window,
                                     int32_t* slot, int64_t n, void* stream) {
  if (n < 0 || window < 1) return PS_ERR_INVALID_ARGUMENT;
  if (n == 0) return PS_OK;
  if (!pos || !prefix_len || !slot) return PS_ERR_INVALID_ARGUMENT;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  ring_slots_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), threads, 0,
                      (cudaStream_t)stream>>>(pos, prefix_len, window, slot, n);
  return launch_status();
}

extern "C" ps_status_t ps_kv_append(const ps_cache_desc* cache, const int32_t* seq_idx,
                                    const int32_t* pos0, const int32_t* cu_tokens, int32_t nrun,
                                    const void* k, const void* v, int64_t n_tokens, void* stream) {
  ps_status_t st = check_cache(cache);
  if (st != PS_OK) return st;
  if (n_tokens < 0 || nrun < 0) return PS_ERR_INVALID_ARGUMENT;
  if (n_tokens == 0) return PS_OK;
  if (nrun < 1 || !seq_idx || !pos0 || !cu_tokens || !k || !v) return PS_ERR_INVALID_ARGUMENT;
  if (!aligned16(k) || !aligned16(v)) return PS_ERR_ALIGNMENT;
  AppendParams p;
  p.k = static_cast<const uint4*>(k);
  p.v = static_cast<const uint4*>(v);
  p.kp = static_cast<uint4*>(cache->k_pool);
  p.vp = static_cast<uint4*>(cache->v_pool);
  p.seq_idx = seq_idx;
  p.pos0 = pos0;
  p.cu = cu_tokens;
  p.slot_base = cache->slot_base;
  p.prefix_len = cache->prefix_len;
  p.status = cache->status;
  p.n_tokens = n_tokens;
  p.total_slots = cache->total_slots;
  p.nrun = nrun;
  p.nseq = cache->nseq;
  p.hkv = cache->n_kv_heads;
  p.head_dim = cache->head_dim;
  p.window = cache->window;
  p.capacity = cache->capacity;
  p.prefix_max = cache->prefix_max;
  make_rope_turns(cache->rope_theta, cache->head_dim, &p.turns);
  const int threads = 256;
  const int64_t items = n_tokens * cache->n_kv_heads * (cache->head_dim / 16);
  int64_t blocks = (items + threads - 1) / threads;
  const int sms = device_sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  append_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(p);
  return launch_status();
}
