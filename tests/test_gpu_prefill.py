"""ps_prefill (RoPE pre-pass + tcgen05 tile kernel) and its tile classes
against the oracle (GPU)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import (FULL, PARTIAL, SKIP, attend, attend_reset_pe, masked_attention, rope, round_bf16,
                    tile_classes, visible_positions)

from _util import (append_runs, assert_attention_close, bf16_tensor_to_f64, bits_to_bf16_tensor,
                   lse_tol_stress, synth_source)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


# ------------------------------------------------------------ tile classes --
def _ring_key_positions(S, q0, P, W):
    n_pre = min(P, q0)
    wlo = max(P, q0 - W)
    return np.array(list(range(n_pre)) + list(range(wlo, q0)) + list(range(q0, q0 + S)))


@pytest.mark.parametrize("S,q0,P,W,ring,bm,bn", [
    (1000, 0, 37, 300, False, 128, 128), (70, 0, 9, 13, False, 16, 8), (97, 0, 30, 5, False, 8, 32),
    (64, 0, 64, 1, False, 16, 16), (300, 700, 20, 64, False, 32, 32), (150, 300, 20, 64, True, 16, 16),
    (150, 50, 20, 64, True, 16, 16), (40, 10, 20, 64, True, 8, 8), (1, 5000, 100, 4096, True, 128, 128),
    (513, 9000, 100, 4096, True, 128, 128), (77, 0, 0, 3, False, 7, 5)])
def test_tile_classes_bit_exact(ps, S, q0, P, W, ring, bm, bn):
    got = ps.prefill_tile_classes(S, q0, P, W, ring, bm, bn).cpu().numpy()
    kpos = _ring_key_positions(S, q0, P, W) if ring else np.arange(q0, q0 + S)
    want = tile_classes(np.arange(q0, q0 + S), kpos, P, W, bm, bn)
    assert np.array_equal(got, want)


def test_tile_classes_full_size_counts(ps):
    g = json.load(open(os.path.join(GOLDEN, "tile_counts.json")))
    for case in g["cases"]:
        got = ps.prefill_tile_classes(case["S"], 0, case["P"], case["W"], False, case["BM"],
                                      case["BN"]).cpu().numpy()
        assert [int((got == k).sum()) for k in (SKIP, PARTIAL, FULL)] == case["skip_partial_full"]
    # and element for element at the prefill workload's size
    pos = np.arange(32768)
    want = tile_classes(pos, pos, 100, 4096, 128, 128)
    assert np.array_equal(ps.prefill_tile_classes(32768, 0, 100, 4096).cpu().numpy(), want)


# ------------------------------------------------------------------ prefill --
def _inputs(seed, B, S, q_start, hq, hkv, D, qscale=0):
    q = np.stack([synth.query_bits(seed, b, np.arange(q_start[b], q_start[b] + S), hq, D, qscale)
                  for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(np.arange(q_start[b], q_start[b] + S))
          for b in range(B)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    return q, k, v


def _run(ps, q, k, v, q_start, P, W, theta, ring=None, pe_mode=None):
    i32 = dict(dtype=torch.int32, device="cuda")
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(bits_to_bf16_tensor(q), bits_to_bf16_tensor(k), bits_to_bf16_tensor(v),
                          torch.tensor(q_start, **i32), torch.tensor(P, **i32), W,
                          rope_theta=theta, ring=ring, status=status, pe_mode=pe_mode)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def _check_rows(seed, out, lse, q, q_start, P, W, theta, rows_per_b, hkv, what="", qs=0,
                reference=attend):
    B = out.shape[0]
    D = out.shape[3]
    for b in range(B):
        hist = synth.History(seed, b, hkv, D)
        ob = out[b]
        def abs_rows(js, hist=hist):
            k_, v_ = hist.rows(js)
            return k_, np.abs(v_)
        for r in rows_per_b[b]:
            p = q_start[b] + r
            qr = synth.bits_to_f64(q[b, r])
            o_ref, l_ref = reference(qr, p, P[b], W, hist.rows, theta)
            # stress cases (q scaled up): the bf16 P V allowance needs sum p|v| / l
            aw = reference(qr, p, P[b], W, abs_rows, theta)[0] if qs else None
            assert_attention_close(bf16_tensor_to_f64(ob[r]), lse[b, :, r].cpu().numpy(), o_ref,
                                   l_ref, f"{what} b={b} row={r}", lse_abs=lse_tol_stress(qs),
                                   abs_weighted=aw)


@pytest.mark.parametrize("B,S,hq,hkv,P,W,qs", [
    (2, 300, 4, 2, [37, 0], 100, 0),     # ragged tail (300 = 2*128 + 44), prefix and band
    (1, 257, 2, 1, [5], 1000, 0),        # W >= S: plain causal
    (1, 384, 2, 2, [0], 128, 0),         # P = 0: vanilla sliding window, tile-aligned W
    (1, 200, 8, 1, [300], 16, 0),        # P >= S: causal through the prefix
    (1, 260, 4, 2, [4], 1, 0),           # W = 1, StreamingLLM-like sink of 4
    (2, 200, 4, 2, [17, 130], 70, 2),    # q x 4: sharper softmax, stale-max rescaling
    (2, 300, 3, 3, [37, 200], 100, 0),   # one query head per KV head: split prefix tile, band
    (1, 333, 6, 2, [150], 90, 0),        # three query heads per KV head (odd group)
    (1, 300, 8, 2, [50], 100, 0),        # four query heads per KV head: two pairs per KV head
])
def test_prefill_all_rows(ps, B, S, hq, hkv, P, W, qs):
    seed, D, theta = 31, 128, 10000.0
    q_start = [0] * B
    q, k, v = _inputs(seed, B, S, q_start, hq, hkv, D, qs)
    out, lse = _run(ps, q, k, v, q_start, P, W, theta)
    _check_rows(seed, out, lse, q, q_start, P, W, theta, [range(S)] * B, hkv, qs=qs)


def _check_all_rows_hoisted(seed, out, lse, q, P, W, theta, hkv, what):
    """Every row of every batch row (chunks at position 0) against the oracle's
    masked attention over the row's visible keys.  The rotation and bf16 rounding
    of each key (which do not depend on the query) are done once per batch row,
    with the oracle's own rope and round_bf16, instead of once per query row."""
    B, S, hq, D = out.shape
    pos = np.arange(S)
    for b in range(B):
        k, v = synth.History(seed, b, hkv, D).rows(pos)
        k_hat = round_bf16(rope(k, pos, theta))
        q_hat = round_bf16(rope(synth.bits_to_f64(q[b]), pos, theta))
        ob = bf16_tensor_to_f64(out[b])
        lb = lse[b].cpu().numpy()
        for r in range(S):
            js = visible_positions(r, P[b], W)
            o_ref, l_ref = masked_attention(q_hat[r], k_hat[js], v[js], 1 / math.sqrt(D))
            assert_attention_close(ob[r], lb[:, r], o_ref, l_ref, f"{what} b={b} row={r}")


@pytest.mark.parametrize("B,S,P", [
    (1, 8192, [100]),       # 64 query tiles x 8 head pairs = 512 work items over the SMs
    (2, 4000, [100, 0]),    # 2 x 32 x 8 = 512 items, a ragged last tile in each batch row
])
def test_prefill_all_rows_several_items_per_cta(ps, B, S, P):
    """The persistent tile kernel gives each CTA three or more work items here, so
    every row checked depends on barrier phases, the Q hand-over and the O
    hand-over carried from item to item."""
    seed, hq, hkv, D, W, theta = 35, 16, 8, 128, 512, 10000.0
    assert B * -(-S // 128) * (hq // 2) >= 3 * torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = _inputs(seed, B, S, [0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0] * B, P, W, theta)
    _check_all_rows_hoisted(seed, out, lse, q, P, W, theta, hkv, "multi-item")


def test_prefill_chunk_without_ring_sees_only_the_chunk(ps):
    """q_start > 0 and no ring: keys are the chunk's own tokens (positions
    q_start..q_start+S-1); the mask is still the absolute-position rule."""
    seed, B, S, hq, hkv, D, P, W, theta = 32, 1, 200, 4, 2, 128, 16, 64, 10000.0
    c0 = 1000
    q, k, v = _inputs(seed, B, S, [c0], hq, hkv, D)
    out, lse = _run(ps, q, k, v, [c0], [P], W, theta)
    hist = synth.History(seed, 0, hkv, D)
    for r in range(S):
        p = c0 + r
        js = visible_positions(p, P, W)
        js = js[js >= c0]
        kr, vv = hist.rows(js)
        qh = round_bf16(rope(synth.bits_to_f64(q[0, r]), p, theta))
        kh = round_bf16(rope(kr, js, theta))
        o_ref, l_ref = masked_attention(qh, kh, vv, 1 / math.sqrt(D))
        assert_attention_close(bf16_tensor_to_f64(out[0, r]), lse[0, :, r].cpu().numpy(), o_ref, l_ref,
                               f"row {r}")


@pytest.mark.parametrize("c0,S,hq", [(300, 150, 4), (50, 150, 4), (10, 40, 4), (5000, 1, 4),
                                     (84, 64, 4), (20, 300, 4), (300, 150, 2), (84, 200, 2)])
def test_prefill_extend_from_ring(ps, c0, S, hq):
    """Chunked extend: the cache holds positions < c0 (after eviction); the
    chunk [c0, c0+S) attends to the ring's live keys plus itself.  hq = 4
    (GQA pairs) and hq = 2 (one query head per KV head) take the two kernels."""
    seed, B, hkv, D, P, W, theta = 33, 2, 2, 128, 20, 64, 10000.0
    cache = ps.RingCache(B, hkv, D, W, [P] * B, rope_theta=theta)
    append_runs(cache, {b: [(0, c0)] for b in range(B)}, synth_source(seed, hkv, D))
    q, k, v = _inputs(seed, B, S, [c0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [c0] * B, [P] * B, W, theta, ring=cache)
    _check_rows(seed, out, lse, q, [c0] * B, [P] * B, W, theta, [range(S)] * B, hkv, "extend")
    assert cache.check_status() == 0


def test_prefill_extend_from_paged_ring(ps):
    """Chunked extend whose cached keys sit in a paged ring (shuffled blocks of 32)."""
    seed, B, hq, hkv, D, P, W, theta, c0, S = 34, 2, 4, 2, 128, 20, 64, 10000.0, 300, 150
    probe = ps.RingCache(B, hkv, D, W, [P] * B, rope_theta=theta, block_size=32, device="cpu")
    order = np.random.default_rng(5).permutation(B * probe.blocks_per_seq)
    cache = ps.RingCache(B, hkv, D, W, [P] * B, rope_theta=theta, block_size=32, block_order=order)
    append_runs(cache, {b: [(0, c0)] for b in range(B)}, synth_source(seed, hkv, D))
    q, k, v = _inputs(seed, B, S, [c0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [c0] * B, [P] * B, W, theta, ring=cache)
    _check_rows(seed, out, lse, q, [c0] * B, [P] * B, W, theta, [range(S)] * B, hkv, "paged extend")
    assert cache.check_status() == 0


def test_prefill_32k_sampled_rows(ps):
    """One Qwen3-1.7B-shaped layer: 32,768 tokens, P = 100, W = 4,096, 16/8
    heads; rows at every boundary of the mask plus random ones."""
    seed, B, S, hq, hkv, D, P, W, theta = 2, 1, 32768, 16, 8, 128, 100, 4096, 10000.0
    q, k, v = _inputs(seed, B, S, [0], hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0], [P], W, theta)
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 99, 100, 127, 128, 4095, 4096, 4196, 4197, 8191, 32767]
                      + list(rng.integers(0, S, 12))))
    _check_rows(seed, out, lse, q, [0], [P], W, theta, [rows], hkv, "32k")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_training_forward_sampled_rows(ps):
    """Truncated-backprop forward: 8 x 8,192 tokens, P = 256, W = 2,048."""
    seed, B, S, hq, hkv, D, P, W, theta = 5, 8, 8192, 16, 8, 128, 256, 2048, 10000.0
    q, k, v = _inputs(seed, B, S, [0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0] * B, [P] * B, W, theta)
    rng = np.random.default_rng(1)
    rows = [sorted(set([0, 255, 256, 2047, 2048, 2303, 8191] + list(rng.integers(0, S, 4))))
            for _ in range(B)]
    _check_rows(seed, out, lse, q, [0] * B, [P] * B, W, theta, rows, hkv, "train")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ---------------------------------------------------------------- Reset PE --
@pytest.mark.parametrize("B,S,hq,hkv,P,W", [
    (2, 400, 4, 2, [37, 128], 64),     # split prefix tile (P % 128 != 0) and a tile-aligned prefix
    (1, 300, 2, 2, [100], 100),        # one query head per KV head (the single-head kernel)
    (1, 520, 4, 2, [200], 30),         # prefix spans two tiles, narrow window
    (2, 260, 4, 2, [0, 300], 50),      # no prefix keys / everything inside the prefix
])
def test_prefill_reset_pe_all_rows(ps, B, S, hq, hkv, P, W):
    """Reset PE: prefix keys see the query rotated at min(p, P + W - 1), window
    keys at p; every row against the oracle's renumbered attention."""
    seed, D, theta = 36, 128, 10000.0
    q, k, v = _inputs(seed, B, S, [0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0] * B, P, W, theta, pe_mode=ps.PS_PE_RESET)
    _check_rows(seed, out, lse, q, [0] * B, P, W, theta, [range(S)] * B, hkv, "reset",
                reference=attend_reset_pe)


def test_prefill_reset_pe_several_items_per_cta(ps):
    """Reset PE through the persistent kernel with several items per CTA (the
    second query load per item): rows at the mask's edges and a random sample."""
    seed, B, S, hq, hkv, D, P, W, theta = 37, 2, 4096, 16, 8, 128, [100, 256], 512, 10000.0
    q, k, v = _inputs(seed, B, S, [0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0] * B, P, W, theta, pe_mode=ps.PS_PE_RESET)
    rng = np.random.default_rng(2)
    rows = [sorted(set([0, 99, 100, 127, 128, 255, 256, 611, 612, 613, 767, 768, 4095]
                       + rng.integers(0, S, 40).tolist())) for _ in range(B)]
    _check_rows(seed, out, lse, q, [0] * B, P, W, theta, rows, hkv, "reset multi-item",
                reference=attend_reset_pe)


@pytest.mark.parametrize("c0,S,hq", [(300, 150, 4), (50, 150, 4), (84, 64, 2), (5000, 130, 4)])
def test_prefill_extend_from_ring_reset_pe(ps, c0, S, hq):
    """Chunked extend against a Reset PE ring: cached keys stay rotated at their
    absolute positions; the chunk's queries are renumbered for the prefix keys."""
    seed, B, hkv, D, P, W, theta = 38, 2, 2, 128, 20, 64, 10000.0
    cache = ps.RingCache(B, hkv, D, W, [P] * B, rope_theta=theta, pe_mode=ps.PS_PE_RESET)
    append_runs(cache, {b: [(0, c0)] for b in range(B)}, synth_source(seed, hkv, D))
    q, k, v = _inputs(seed, B, S, [c0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [c0] * B, [P] * B, W, theta, ring=cache)
    _check_rows(seed, out, lse, q, [c0] * B, [P] * B, W, theta, [range(S)] * B, hkv,
                "reset extend", reference=attend_reset_pe)
    assert cache.check_status() == 0


# ------------------------------------------------------------- head_dim 64 --
@pytest.mark.parametrize("B,S,hq,hkv,P,W,pe", [
    (2, 300, 4, 2, [37, 0], 100, 0),     # pairs of query heads, ragged tail
    (1, 257, 2, 2, [5], 1000, 0),        # one query head per KV head; W >= S
    (1, 400, 4, 2, [37], 64, 1),         # Reset PE with a split prefix tile
])
def test_prefill_head_dim_64_all_rows(ps, B, S, hq, hkv, P, W, pe):
    seed, D, theta = 39, 64, 10000.0
    q, k, v = _inputs(seed, B, S, [0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [0] * B, P, W, theta, pe_mode=pe)
    _check_rows(seed, out, lse, q, [0] * B, P, W, theta, [range(S)] * B, hkv, "D=64",
                reference=attend_reset_pe if pe else attend)


def test_prefill_head_dim_64_extend_from_ring(ps):
    seed, B, hq, hkv, D, P, W, theta, c0, S = 40, 2, 4, 2, 64, 20, 64, 10000.0, 300, 150
    cache = ps.RingCache(B, hkv, D, W, [P] * B, rope_theta=theta)
    append_runs(cache, {b: [(0, c0)] for b in range(B)}, synth_source(seed, hkv, D))
    q, k, v = _inputs(seed, B, S, [c0] * B, hq, hkv, D)
    out, lse = _run(ps, q, k, v, [c0] * B, [P] * B, W, theta, ring=cache)
    _check_rows(seed, out, lse, q, [c0] * B, [P] * B, W, theta, [range(S)] * B, hkv, "D=64 extend")
    assert cache.check_status() == 0


def test_prefill_extend_ragged_chunks_through_ring_seq(ps):
    """Three batch rows extend three of four cached sequences, chosen through
    ring_seq (not in order), each at its own chunk start and with its own prefix:
    inside the prefix, just past P + W, and long after (with eviction)."""
    seed, hq, hkv, D, W, theta, S = 45, 4, 2, 128, 64, 10000.0, 160
    P_seq = [20, 5, 40, 0]            # prefix of each cached sequence
    c0_seq = [900, 30, 110, 400]      # positions already cached per sequence
    cache = ps.RingCache(4, hkv, D, W, P_seq, rope_theta=theta)
    append_runs(cache, {s: [(0, c0_seq[s])] for s in range(4)}, synth_source(seed, hkv, D))
    rows = [2, 0, 1]                  # batch row b extends sequence rows[b]
    c0 = [c0_seq[s] for s in rows]
    P = [P_seq[s] for s in rows]
    B = len(rows)
    q = np.stack([synth.query_bits(seed, s, np.arange(c0[b], c0[b] + S), hq, D)
                  for b, s in enumerate(rows)])
    kv = [synth.History(seed, s, hkv, D).rows_bits(np.arange(c0[b], c0[b] + S))
          for b, s in enumerate(rows)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    i32 = dict(dtype=torch.int32, device="cuda")
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(bits_to_bf16_tensor(q), bits_to_bf16_tensor(k), bits_to_bf16_tensor(v),
                          torch.tensor(c0, **i32), torch.tensor(P, **i32), W, rope_theta=theta,
                          ring=cache, ring_seq=torch.tensor(rows, **i32), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and cache.check_status() == 0
    for b, s in enumerate(rows):
        hist = synth.History(seed, s, hkv, D)
        for r in range(S):
            o_ref, l_ref = attend(synth.bits_to_f64(q[b, r]), c0[b] + r, P[b], W, hist.rows, theta)
            assert_attention_close(bf16_tensor_to_f64(out[b, r]), lse[b, :, r].cpu().numpy(), o_ref,
                                   l_ref, f"b={b} (sequence {s}) row={r}")


@pytest.mark.parametrize("hq,hkv", [(4, 2), (3, 3)])
def test_prefill_output_only_16_byte_aligned(ps, hq, hkv):
    """An output buffer that is 16- but not 32-byte aligned takes the 16-byte store
    path and gives the same bits as an aligned one (pair and odd-group kernels)."""
    seed, B, S, D, W, theta = 41, 1, 300, 128, 100, 10000.0
    P, q_start = [37], [0]
    q, k, v = _inputs(seed, B, S, q_start, hq, hkv, D)
    i32 = dict(dtype=torch.int32, device="cuda")
    args = (bits_to_bf16_tensor(q), bits_to_bf16_tensor(k), bits_to_bf16_tensor(v),
            torch.tensor(q_start, **i32), torch.tensor(P, **i32), W)
    ref, ref_lse = ps.prefill(*args, rope_theta=theta)
    n = B * S * hq * D
    raw = torch.zeros(n + 64, dtype=torch.bfloat16, device="cuda")
    off = next(o for o in range(0, 64, 8) if (raw.data_ptr() + 2 * o) % 32 == 16)
    out = raw[off:off + n].view(B, S, hq, D)
    assert out.data_ptr() % 32 == 16
    got, got_lse = ps.prefill(*args, rope_theta=theta, out=out)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse)
    assert torch.count_nonzero(raw[:off]).item() == 0 and torch.count_nonzero(raw[off + n:]).item() == 0
