"""Seeded, counter-based synthetic inputs shared by the oracle and the CUDA tests.

This module holds no attention, RoPE or cache arithmetic: it only turns a
(seed, stream, seq, pos, head, dim) coordinate into a standard-normal value
rounded to bfloat16.  Because every value is a pure function of its
coordinate, any slice of an arbitrarily long K/V history can be produced on
demand without materialising the rest of it.

Definition
----------
* Counter: ``idx = ((seq * 2**20 + pos) * 64 + head) * 256 + dim`` (requires
  seq < 2**12, pos < 2**20, head < 64, dim < 256).
* Key: ``key = splitmix64(seed * 2**8 + stream)``.
* Two uniforms: ``u_i = ((splitmix64(key ^ (2*idx + i)) >> 11) + 0.5) * 2**-53``
  for i = 0, 1, with ``splitmix64`` the published SplitMix64 output function
  (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; constants as in Vigna's reference ``splitmix64.c``).
* Normal: Box-Muller, ``z = sqrt(-2 ln u_0) * cos(2 pi u_1)`` in float64.
* Storage: ``z`` is cast to float32 (round to nearest even), then to bfloat16
  (round to nearest even on the float32 bits).  Arrays are returned as uint16
  bit patterns; ``bits_to_f64`` decodes them.

Streams: Q=0, K=1, V=2 (others free for the caller).
"""
from __future__ import annotations

import numpy as np

STREAM_Q = 0
STREAM_K = 1
STREAM_V = 2

def _splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function; arithmetic wraps modulo 2**64 by design."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode uint16 bfloat16 bit patterns to float64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def normal_bf16(seed: int, stream: int, seq, pos, heads: int, dim: int) -> np.ndarray:
    """Standard-normal bfloat16 bits for coordinates (seq, pos) x [heads] x [dim].

    ``seq`` and ``pos`` are broadcast against each other (scalars or 1-D arrays of
    equal length).  Returns uint16 of shape ``[n, heads, dim]``.
    """
    seq = np.atleast_1d(np.asarray(seq, dtype=np.int64))
    pos = np.atleast_1d(np.asarray(pos, dtype=np.int64))
    seq, pos = np.broadcast_arrays(seq, pos)
    if seq.size and (seq.min() < 0 or seq.max() >= 1 << 12):
        raise ValueError("seq out of range [0, 4096)")
    if pos.size and (pos.min() < 0 or pos.max() >= 1 << 20):
        raise ValueError("pos out of range [0, 2**20)")
    if not (0 < heads <= 64 and 0 < dim <= 256):
        raise ValueError("heads/dim out of range")
    rows_per_chunk = max(1, (1 << 22) // (heads * dim))
    if seq.size > rows_per_chunk:  # bound the temporaries of large requests
        return np.concatenate([normal_bf16(seed, stream, seq[i:i + rows_per_chunk],
                                           pos[i:i + rows_per_chunk], heads, dim)
                               for i in range(0, seq.size, rows_per_chunk)])
    key = _splitmix64(np.uint64(seed * 256 + stream))
    row = (seq.astype(np.uint64) << np.uint64(20)) + pos.astype(np.uint64)
    h = np.arange(heads, dtype=np.uint64)
    d = np.arange(dim, dtype=np.uint64)
    idx = ((row[:, None, None] * np.uint64(64) + h[None, :, None]) * np.uint64(256)
           + d[None, None, :])
    u0 = _splitmix64(key ^ (idx * np.uint64(2)))
    u1 = _splitmix64(key ^ (idx * np.uint64(2) + np.uint64(1)))
    scale = 2.0 ** -53
    f0 = ((u0 >> np.uint64(11)).astype(np.float64) + 0.5) * scale
    f1 = ((u1 >> np.uint64(11)).astype(np.float64) + 0.5) * scale
    z = np.sqrt(-2.0 * np.log(f0)) * np.cos(2.0 * np.pi * f1)
    return f32_to_bf16_bits(z.astype(np.float32))


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive), from the same counter scheme."""
    key = _splitmix64(np.uint64(seed * 256 + stream))
    z = _splitmix64(key ^ np.arange(n, dtype=np.uint64))
    span = np.uint64(hi - lo + 1)
    return (z % span).astype(np.int64) + lo


class History:
    """On-demand raw (pre-RoPE) K/V history of one synthetic sequence.

    ``rows(pos)`` returns float64 arrays ``k, v`` of shape [len(pos), heads, dim]
    holding the raw bfloat16 values at the given absolute positions.
    """

    def __init__(self, seed: int, seq: int, heads: int, dim: int):
        self.seed, self.seq, self.heads, self.dim = seed, seq, heads, dim

    def rows_bits(self, pos):
        k = normal_bf16(self.seed, STREAM_K, self.seq, pos, self.heads, self.dim)
        v = normal_bf16(self.seed, STREAM_V, self.seq, pos, self.heads, self.dim)
        return k, v

    def rows(self, pos):
        k, v = self.rows_bits(pos)
        return bits_to_f64(k), bits_to_f64(v)


def query_bits(seed: int, seq, pos, heads: int, dim: int, qscale_log2: int = 0) -> np.ndarray:
    """Raw query bits; ``qscale_log2`` multiplies by an exact power of two."""
    b = normal_bf16(seed, STREAM_Q, seq, pos, heads, dim)
    if qscale_log2:
        x = bits_to_f64(b) * (2.0 ** qscale_log2)
        b = f32_to_bf16_bits(x.astype(np.float32))
    return b
