// ps_ring.cu -- ring-slot mapping and the RoPE + append kernel.
//
// The cache keeps P fixed prefix slots and W rotating window slots per
// sequence (njhaofan.com section "PrefixSliding如何丢掉中间Token？"; the
// "伪代码" section of the papers.ananclaw.com explainer fixes the cache size at
// prefix_len + W).  Keys are rotated once, at their absolute position, when
// they are appended, and never again (Continue PE, agihunt.info paragraph on
// position encodings).
#include "ps_internal.h"
#include "ps_rope.cuh"

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
  const int32_t* prefix_len;
  int32_t* status;
  SlotMap map;
  int64_t n_tokens;
  int32_t nrun, nseq, hkv, head_dim, window, prefix_max;
  RopeTurns turns;
};

// A block of 128 threads takes 128 / (D/2) tokens at a time.  First each
// thread resolves one (token, rotation pair): the token's run, sequence,
// position and destination row, and the (cos, sin) of the pair's angle, into
// shared memory; the angle of a position is shared by all KV heads.  Then one
// thread per (token, kv head, group of 8 pairs) loads the 8 elements of the
// first half and their 8 partners (two 16-byte loads), rotates them in fp32 and
// stores bf16 (round to nearest even); V is copied alongside.
constexpr int kAppendThreads = 128;

constexpr int kAppendCuSmem = 2048;  // run offsets staged in shared memory up to this many

__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AppendParams p) {
  __shared__ float2 cs[kAppendThreads];
  __shared__ int64_t row_of[kAppendThreads];  // destination pool row, or -1 = write nothing
  __shared__ int32_t s_cu[kAppendCuSmem];
  grid_dependency_wait();  // inputs and the pool may be in use by earlier stream work
  allow_dependents();
  // the run lookup below is a binary search over cu: in shared memory it costs a
  // few cycles per step instead of a dependent global load per step
  const bool cu_in_smem = p.nrun + 1 <= kAppendCuSmem;
  if (cu_in_smem) {
    for (int i = threadIdx.x; i <= p.nrun; i += kAppendThreads) s_cu[i] = p.cu[i];
    __syncthreads();
  }
  const int32_t* cu = cu_in_smem ? s_cu : p.cu;
  const int half = p.head_dim / 2;
  const int tpb = kAppendThreads / half;     // tokens per block iteration
  const int groups = p.head_dim / 16;
  const int vec_per_row = p.head_dim / 8;    // 16-byte vectors per head row
  const int64_t n_groups = (p.n_tokens + tpb - 1) / tpb;
  for (int64_t tg = blockIdx.x; tg < n_groups; tg += gridDim.x) {
    {
      const int tl = threadIdx.x / half, i = threadIdx.x % half;
      const int64_t t = tg * tpb + tl;
      int64_t row = -1;
      int32_t pos = 0;
      if (t < p.n_tokens) {
        // run r: the largest r with cu[r] <= t
        int lo = 0, hi = p.nrun - 1;
        while (lo < hi) {
          int mid = (lo + hi + 1) >> 1;
          if (cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int64_t c0 = cu[lo], c1 = cu[lo + 1];
        const int32_t s = p.seq_idx[lo];
        int32_t bad = 0;
        if (!(c0 <= t && t < c1)) bad = PS_DEV_BAD_RUN;
        else if (s < 0 || s >= p.nseq) bad = PS_DEV_BAD_SEQ;
        int32_t P = 0;
        int64_t last = 0;
        if (!bad) {
          P = p.prefix_len[s];
          const int64_t first = p.pos0[lo];
          last = first + (c1 - c0) - 1;
          if (P < 0 || P > p.prefix_max) bad = PS_DEV_BAD_PREFIX;
          else if (!p.map.seq_ok(s)) bad = PS_DEV_BAD_SLOT;
          else if (first < 0 || last > 0x7fffffffLL) bad = PS_DEV_BAD_POS;
          else pos = (int32_t)(first + (t - c0));
        }
        if (!bad && (pos < P || (int64_t)pos > last - p.window)) {
          // a window position is overwritten later in the same run once a
          // position W further on is also in it: only prefix positions and
          // the last W of the run survive
          row = p.map.row(s, ring_slot(pos, P, p.window));
          if (row < 0) bad = PS_DEV_BAD_SLOT;
        }
        if (bad && i == 0) set_flag(p.status, bad);
      }
      float c = 1.f, sn = 0.f;
      if (row >= 0) rope_cos_sin(pos, p.turns.f[i], c, sn);
      cs[threadIdx.x] = make_float2(c, sn);
      if (i == 0) row_of[tl] = row;
    }
    __syncthreads();
    const int items = tpb * p.hkv * groups;
    for (int it = threadIdx.x; it < items; it += kAppendThreads) {
      const int g = it % groups;
      const int h = (it / groups) % p.hkv;
      const int tl = it / (groups * p.hkv);
      const int64_t row = row_of[tl];
      if (row < 0) continue;
      const int64_t t = tg * tpb + tl;
      const int64_t src = (t * p.hkv + h) * vec_per_row;
      const int64_t dst = (row * p.hkv + h) * vec_per_row;
      const int half_vec = vec_per_row / 2;
      const float2* ang = &cs[tl * half + 8 * g];
      uint4 a = p.k[src + g], b = p.k[src + half_vec + g];
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
      const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b);
      uint4 ra, rb;
      uint32_t* raw = reinterpret_cast<uint32_t*>(&ra);
      uint32_t* rbw = reinterpret_cast<uint32_t*>(&rb);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 t0 = ang[2 * e], t1 = ang[2 * e + 1];
        const float x0 = bf16lo(aw[e]), x1 = bf16hi(aw[e]);  // first-half elements
        const float y0 = bf16lo(bw[e]), y1 = bf16hi(bw[e]);  // their partners
        raw[e] = pack_bf16(rope_first(x0, y0, t0.x, t0.y), rope_first(x1, y1, t1.x, t1.y));
        rbw[e] = pack_bf16(rope_second(x0, y0, t0.x, t0.y), rope_second(x1, y1, t1.x, t1.y));
      }
      p.kp[dst + g] = ra;
      p.kp[dst + half_vec + g] = rb;
      p.vp[dst + g] = p.v[src + g];
      p.vp[dst + half_vec + g] = p.v[src + half_vec + g];
    }
    __syncthreads();
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
  p.prefix_len = cache->prefix_len;
  p.status = cache->status;
  p.map = slot_map(cache);
  p.n_tokens = n_tokens;
  p.nrun = nrun;
  p.nseq = cache->nseq;
  p.hkv = cache->n_kv_heads;
  p.head_dim = cache->head_dim;
  p.window = cache->window;
  p.prefix_max = cache->prefix_max;
  make_rope_turns(cache->rope_theta, cache->head_dim, &p.turns);
  const int64_t tpb = kAppendThreads / (cache->head_dim / 2);
  int64_t blocks = (n_tokens + tpb - 1) / tpb;
  const int sms = device_sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  if (launch_dependent(append_kernel, dim3((unsigned)blocks), dim3(kAppendThreads), 0,
                       (cudaStream_t)stream, p) != cudaSuccess)
    return PS_ERR_CUDA;
  return launch_status();
}

extern "C" ps_status_t ps_device_code_version(int32_t* version) {
  if (!version) return PS_ERR_INVALID_ARGUMENT;
  cudaFuncAttributes a;
  if (cudaFuncGetAttributes(&a, ring_slots_kernel) != cudaSuccess) {
    cudaGetLastError();
    return PS_ERR_CUDA;
  }
  *version = a.binaryVersion;
  return PS_OK;
}
