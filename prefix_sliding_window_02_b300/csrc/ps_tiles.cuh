// ps_tiles.cuh -- key-position map and tile classes for the prefill kernel.
//
// Two-level filter of the FlashAttention kernel ("Prefix Sliding for efficient
// test-time scaling", agihunt.info, paragraph on the kernel; njhaofan.com
// section "PrefixSliding如何丢掉中间Token？"): a tile that holds no admitted
// (query, key) pair is skipped, a tile that holds some is masked element by
// element, a tile whose pairs are all admitted runs unmasked.
//
// Keys of one batch row sit in an array whose positions are two increasing
// runs: indices [0, n_pre) hold positions 0..n_pre-1 (the cached prefix) and
// indices [n_pre, n_keys) hold positions base2, base2+1, ... (cached window,
// then the chunk).  Without a ring n_pre = 0 and base2 = q_start.
#pragma once

#include <stdint.h>

namespace ps {

enum : uint8_t { kSkip = 0, kPartial = 1, kFull = 2 };

struct KeyMap {
  int32_t n_pre;   // keys in the first run
  int32_t base2;   // position of key index n_pre
  int32_t n_keys;  // total keys
};

// Key array a chunk [q_start, q_start + seqlen) sees.  With a ring, the ring
// holds what query q_start-1 may see: positions < min(P, q_start) and the
// window positions [max(P, q_start - W), q_start).
__host__ __device__ inline KeyMap make_keymap(int32_t seqlen, int32_t q_start, int32_t P,
                                              int32_t W, bool with_ring) {
  KeyMap m;
  if (!with_ring) {
    m.n_pre = 0;
    m.base2 = q_start;
    m.n_keys = seqlen;
    return m;
  }
  const int32_t n_pre = q_start < P ? q_start : P;
  const int32_t wlo = (q_start - W) > P ? (q_start - W) : P;
  const int32_t n_win = q_start > wlo ? q_start - wlo : 0;
  m.n_pre = n_pre;
  m.base2 = q_start - n_win;
  m.n_keys = n_pre + n_win + seqlen;
  return m;
}

__host__ __device__ inline int32_t key_pos(const KeyMap& m, int32_t k) {
  return k < m.n_pre ? k : m.base2 + (k - m.n_pre);
}

// Number of keys whose position is < x.
__host__ __device__ inline int32_t keys_below(const KeyMap& m, int64_t x) {
  int64_t a = x < 0 ? 0 : (x > m.n_pre ? m.n_pre : x);
  int64_t r = x - m.base2;
  const int64_t n2 = m.n_keys - m.n_pre;
  int64_t b = r < 0 ? 0 : (r > n2 ? n2 : r);
  return (int32_t)(a + b);
}

__host__ __device__ inline bool admitted(int64_t p, int64_t j, int32_t P, int32_t W) {
  return j <= p && (j < P || j > p - W);
}

// Some query in [q0, q1] admits some key position in [j0, j1]?
__host__ __device__ inline bool interval_any(int64_t q0, int64_t q1, int64_t j0, int64_t j1,
                                             int32_t P, int32_t W) {
  if (j0 > j1) return false;
  if (j0 < P && j0 <= q1) return true;                    // a prefix key
  const int64_t lo = q0 > j0 ? q0 : j0;                    // a window key
  const int64_t hi = q1 < j1 + W - 1 ? q1 : j1 + W - 1;
  return lo <= hi;
}

// Every query in [q0, q1] admits every key position in [j0, j1]?
__host__ __device__ inline bool interval_all(int64_t q0, int64_t q1, int64_t j0, int64_t j1,
                                             int32_t P, int32_t W) {
  if (j0 > j1) return true;
  if (j1 > q0) return false;                               // some key after some query
  if (j1 < P) return true;                                 // all prefix keys
  const int64_t first_window = j0 > P ? j0 : P;            // smallest non-prefix key
  return first_window > q1 - W;                            // still in the last query's window
}

// Class of the tile: query rows [qa, qb] (array order, positions q_start + row),
// key indices [ka, kb] (clipped to the key array).
__host__ __device__ inline uint8_t tile_class(const KeyMap& m, int32_t q_start, int32_t qa,
                                              int32_t qb, int32_t ka, int32_t kb, int32_t P,
                                              int32_t W) {
  const int64_t q0 = (int64_t)q_start + qa, q1 = (int64_t)q_start + qb;
  // split the key indices at the run boundary
  int64_t a0 = 1, a1 = 0, b0 = 1, b1 = 0;  // empty intervals
  if (ka < m.n_pre) {
    a0 = ka;
    a1 = kb < m.n_pre ? kb : m.n_pre - 1;
  }
  if (kb >= m.n_pre) {
    const int32_t s = ka > m.n_pre ? ka : m.n_pre;
    b0 = key_pos(m, s);
    b1 = key_pos(m, kb);
  }
  const bool any = interval_any(q0, q1, a0, a1, P, W) || interval_any(q0, q1, b0, b1, P, W);
  if (!any) return kSkip;
  const bool all = interval_all(q0, q1, a0, a1, P, W) && interval_all(q0, q1, b0, b1, P, W);
  return all ? kFull : kPartial;
}

}  // namespace ps
