"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a library routine, a closed form, a
value printed on the pages, or an independent brute-force enumeration, so that
a dropped term, a wrong sign, index or operand fails somewhere here.
"""
import cmath
import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import (FULL, PARTIAL, SKIP, RingSim, allowed, attend, masked_attention,
                    ring_slot, rope, round_bf16, tile_classes, visible_positions)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- bf16 ----
def test_round_bf16_matches_torch_cast_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 120, 200000))).astype(np.float32)
    x = np.concatenate([x, np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 2**-130, 3e38], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_bf16_ties_to_even_by_hand():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1.
    assert round_bf16(1 + 2**-8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: the even one is 1 + 2^-6.
    assert round_bf16(1 + 3 * 2**-8) == 1 + 2**-6
    # just above a tie rounds up (float64 input, single rounding)
    assert round_bf16(1 + 2**-8 + 2**-30) == 1 + 2**-7
    assert round_bf16(0.0) == 0.0


def test_synth_bf16_cast_matches_torch():
    x = np.random.default_rng(2).standard_normal(100000).astype(np.float32)
    got = synth.bits_to_f64(synth.f32_to_bf16_bits(x))
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)


def test_synth_is_standard_normal_and_coordinate_pure():
    a = synth.bits_to_f64(synth.normal_bf16(3, synth.STREAM_K, 0, np.arange(4000), 4, 64))
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    # any slice equals the same slice generated alone
    b = synth.bits_to_f64(synth.normal_bf16(3, synth.STREAM_K, 0, [17, 3999], 4, 64))
    assert np.array_equal(b, a[[17, 3999]])


# ----------------------------------------------------------------- RoPE ----
def test_rope_identity_at_position_zero():
    x = np.random.default_rng(3).standard_normal((5, 128))
    assert np.allclose(rope(x, 0, 10000.0), x, atol=0, rtol=0)


def test_rope_hand_computed_d4():
    # D = 4, theta = 100: pairs (0,2) at frequency 1 and (1,3) at 100^(-1/2) = 0.1.
    p = 7
    x = np.array([1.0, 2.0, 3.0, 4.0])
    a0, a1 = p * 1.0, p * 0.1
    want = np.array([1 * math.cos(a0) - 3 * math.sin(a0),
                     2 * math.cos(a1) - 4 * math.sin(a1),
                     3 * math.cos(a0) + 1 * math.sin(a0),
                     4 * math.cos(a1) + 2 * math.sin(a1)])
    assert np.allclose(rope(x, p, 100.0), want, rtol=1e-15, atol=1e-15)


def test_rope_as_complex_rotation():
    # Independent form: element pair (i, i+D/2) is the complex number x_i + i x_{i+D/2}
    # multiplied by exp(i * pos * theta^(-2i/D)).
    rng = np.random.default_rng(4)
    d, theta = 16, 10000.0
    for pos in (1, 1000, 262143):
        x = rng.standard_normal(d)
        got = rope(x, pos, theta)
        for i in range(d // 2):
            z = complex(x[i], x[i + d // 2]) * cmath.exp(1j * pos * theta ** (-2 * i / d))
            assert abs(got[i] - z.real) < 1e-12 and abs(got[i + d // 2] - z.imag) < 1e-12


def test_rope_norm_and_relative_position_invariance():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p, j, shift in ((100, 40, 131072), (5000, 4999, 7), (262143, 0, 1)):
        assert abs(np.linalg.norm(rope(q, p, 1e4)) - np.linalg.norm(q)) < 1e-12
        a = rope(q, p, 1e4) @ rope(k, j, 1e4)
        b = rope(q, p + shift, 1e4) @ rope(k, j + shift, 1e4)
        assert abs(a - b) < 1e-9


def test_rope_per_row_positions_broadcast():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 2, 8))
    pos = np.array([0, 5, 9])
    got = rope(x, pos, 1e4)
    for r in range(3):
        assert np.allclose(got[r], rope(x[r], pos[r], 1e4))


# ----------------------------------------------------------------- mask ----
def test_key_count_closed_form_bruteforce():
    for S in range(1, 17):
        for P in range(0, S + 1):
            for W in range(1, S + 2):
                for p in range(S):
                    n = len(visible_positions(p, P, W))
                    assert n == min(p + 1, P + W), (S, P, W, p)


def test_pages_cap_4196_keys():
    g = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))
    c = g["cap_prefix100_window4096"]
    for p in (4195, 4196, 100000, 262143):
        assert len(visible_positions(p, c["P"], c["W"])) <= c["max_keys"]
    assert len(visible_positions(100000, c["P"], c["W"])) == c["max_keys"]


def test_mask_contains_prefix_and_current_token():
    vis = visible_positions(100000, 100, 4096)
    assert vis[0] == 0 and vis[99] == 99 and vis[100] == 100000 - 4095 and vis[-1] == 100000


# ------------------------------------------------------- masked softmax ----
def _sdpa_rows(qh, kh, vh, mask):
    """torch SDPA in float64. qh [S,Hq,D], kh/vh [S,Hkv,D], mask [S,S] bool."""
    hq, hkv = qh.shape[1], kh.shape[1]
    g = hq // hkv
    q = torch.from_numpy(qh).permute(1, 0, 2)
    k = torch.from_numpy(kh).permute(1, 0, 2).repeat_interleave(g, 0)
    v = torch.from_numpy(vh).permute(1, 0, 2).repeat_interleave(g, 0)
    m = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m)
    sc = (q @ k.transpose(1, 2)) / math.sqrt(qh.shape[2])
    lse = torch.logsumexp(sc.masked_fill(~m, -math.inf), dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("S,P,W", [(40, 40, 64), (40, 0, 9), (40, 4, 9), (33, 7, 1), (50, 12, 16)])
def test_attend_matches_sdpa_with_explicit_mask(S, P, W):
    seed, hq, hkv, d, theta = 11, 4, 2, 32, 10000.0
    hist = synth.History(seed, 0, hkv, d)
    pos = np.arange(S)
    q_raw = synth.bits_to_f64(synth.query_bits(seed, 0, pos, hq, d))
    k_raw, v = hist.rows(pos)
    qh = round_bf16(rope(q_raw, pos, theta))
    kh = round_bf16(rope(k_raw, pos, theta))
    jj, pp = np.meshgrid(pos, pos)
    if W >= S:   # reduction 1: no sliding at all -> plain causal
        mask = jj <= pp
    elif P == 0:  # reduction 2: no prefix -> plain band (vanilla sliding window)
        mask = (jj <= pp) & (jj > pp - W)
    else:        # prefix rows OR band, built as the union of two textbook masks
        mask = ((jj <= pp) & (jj < P)) | ((jj <= pp) & (jj > pp - W))
    o_ref, lse_ref = _sdpa_rows(qh, kh, v, mask)
    for p in range(S):
        o, lse = attend(q_raw[p], p, P, W, hist.rows, theta)
        assert np.allclose(o, o_ref[p], atol=1e-12, rtol=1e-10)
        assert np.allclose(lse, lse_ref[p], atol=1e-12, rtol=1e-12)


def test_masked_attention_one_key_and_uniform_keys():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((4, 16))
    k = rng.standard_normal((1, 2, 16))
    v = rng.standard_normal((1, 2, 16))
    o, lse = masked_attention(q, k, v, 0.25)
    for h in range(4):
        assert np.allclose(o[h], v[0, h // 2], rtol=0, atol=0)
        assert abs(lse[h] - 0.25 * (q[h] @ k[0, h // 2])) < 1e-14
    n = 37
    ku = np.repeat(k, n, axis=0)
    vu = rng.standard_normal((n, 2, 16))
    o, lse = masked_attention(q, ku, vu, 0.25)
    for h in range(4):
        assert np.allclose(o[h], vu[:, h // 2].mean(0), atol=1e-14)
        assert abs(lse[h] - (math.log(n) + 0.25 * (q[h] @ k[0, h // 2]))) < 1e-12


def test_attend_zero_keys_gives_mean_of_visible_values():
    # raw k = 0 -> every score is 0 -> O = mean(V over visible keys), LSE = ln(count)
    d, hkv = 16, 1
    rng = np.random.default_rng(8)
    vals = rng.standard_normal((300, hkv, d))

    def hist(js):
        return np.zeros((len(js), hkv, d)), vals[js]

    for (p, P, W) in ((0, 5, 3), (10, 5, 3), (299, 16, 32), (299, 0, 7), (40, 100, 4)):
        o, lse = attend(rng.standard_normal((2, d)), p, P, W, hist, 1e4)
        js = [j for j in range(p + 1) if j < P or j > p - W]
        assert np.allclose(o[0], vals[js, 0].mean(0), atol=1e-13)
        assert abs(lse[0] - math.log(min(p + 1, P + W))) < 1e-13


def _bruteforce_attend(q_raw, p, P, W, hist, theta):
    """Scalar Python: key set as a union of two ranges, RoPE as a complex
    rotation, bf16 by frexp, softmax without max subtraction."""
    def bf16(x):
        if x == 0.0:
            return 0.0
        m, e = math.frexp(x)
        return math.ldexp(round(m * 256), e - 8)

    def rot(vec, pos):
        d = len(vec)
        out = [0.0] * d
        for i in range(d // 2):
            z = complex(vec[i], vec[i + d // 2]) * cmath.exp(1j * pos * theta ** (-2 * i / d))
            out[i], out[i + d // 2] = bf16(z.real), bf16(z.imag)
        return out

    keys = sorted(set(range(0, min(P, p + 1))) | set(range(max(0, p - W + 1), p + 1)))
    k_raw, v = hist(np.array(keys))
    hq, d = q_raw.shape
    hkv = k_raw.shape[1]
    outs, lses = [], []
    for h in range(hq):
        qv = rot(list(q_raw[h]), p)
        ws, acc = [], [0.0] * d
        for n, j in enumerate(keys):
            kv = rot(list(k_raw[n, h * hkv // hq]), j)
            ws.append(math.exp(sum(a * b for a, b in zip(qv, kv)) / math.sqrt(d)))
        tot = sum(ws)
        for n in range(len(keys)):
            for t in range(d):
                acc[t] += ws[n] / tot * v[n, h * hkv // hq, t]
        outs.append(acc)
        lses.append(math.log(tot))
    return np.array(outs), np.array(lses)


def test_attend_matches_pure_python_enumeration_on_tiny_inputs():
    seed, hq, hkv, d, theta = 21, 2, 1, 8, 10000.0
    hist = synth.History(seed, 1, hkv, d)
    for S in (5, 12):
        q_raw = synth.bits_to_f64(synth.query_bits(seed, 1, np.arange(S), hq, d))
        for P in range(0, S + 1):
            for W in range(1, S + 2):
                for p in range(S):
                    o, lse = attend(q_raw[p], p, P, W, hist.rows, theta)
                    ob, lb = _bruteforce_attend(q_raw[p], p, P, W, hist.rows, theta)
                    assert np.allclose(o, ob, atol=1e-12), (S, P, W, p)
                    assert np.allclose(lse, lb, atol=1e-12), (S, P, W, p)


# ----------------------------------------------------------------- ring ----
@pytest.mark.parametrize("P,W,steps", [(16, 32, 4352), (0, 5, 300), (3, 1, 200), (100, 4096, 9000), (64, 8, 500)])
def test_ring_live_set_equals_mask_after_every_append(P, W, steps):
    ring = RingSim(P, W)
    for p in range(steps):
        s = ring.append(p)
        assert 0 <= s < P + W
        ring.check(p)


def test_ring_slot_of_prefix_and_first_window_is_identity():
    for P, W in ((16, 32), (0, 7), (100, 4096)):
        for pos in range(P + W):
            assert ring_slot(pos, P, W) == pos
        # after wrap-around, pos and pos + W share a slot
        assert ring_slot(P + W + 3, P, W) == ring_slot(P + 3, P, W)


# ---------------------------------------------------------------- tiles ----
def _classes_by_intervals(q_pos, k_pos, P, W, BM, BN):
    """Independent classification: each query row admits keys in
    [0, min(P, p+1)) U [max(0, p-W+1), p]; count admitted keys per tile by
    interval arithmetic (key positions must be consecutive)."""
    nq, nk = -(-len(q_pos) // BM), -(-len(k_pos) // BN)
    out = np.zeros((nq, nk), dtype=np.uint8)
    for a in range(nq):
        rows = q_pos[a * BM:(a + 1) * BM]
        for b in range(nk):
            k0, k1 = k_pos[b * BN], k_pos[min((b + 1) * BN, len(k_pos)) - 1]
            tot, n = 0, (k1 - k0 + 1)
            for p in rows:
                lo1, hi1 = 0, min(P, p + 1) - 1
                lo2, hi2 = max(0, p - W + 1), p
                c1 = max(0, min(hi1, k1) - max(lo1, k0) + 1)
                c2 = max(0, min(hi2, k1) - max(lo2, k0) + 1)
                ov = max(0, min(hi1, hi2, k1) - max(lo1, lo2, k0) + 1)
                tot += c1 + c2 - ov
            out[a, b] = SKIP if tot == 0 else (FULL if tot == n * len(rows) else PARTIAL)
    return out


@pytest.mark.parametrize("S,q0,P,W,BM,BN", [(70, 0, 9, 13, 16, 16), (70, 0, 0, 70, 16, 8), (97, 0, 30, 5, 8, 32),
                                            (64, 0, 64, 1, 16, 16), (50, 0, 3, 200, 32, 32)])
def test_tile_classes_match_interval_counting(S, q0, P, W, BM, BN):
    pos = np.arange(q0, q0 + S)
    assert np.array_equal(tile_classes(pos, pos, P, W, BM, BN), _classes_by_intervals(pos, pos, P, W, BM, BN))


def test_tile_classes_causal_closed_form():
    # W >= S, P = 0, square tiles: below the diagonal FULL, on it PARTIAL, above SKIP.
    pos = np.arange(64)
    c = tile_classes(pos, pos, 0, 64, 16, 16)
    for a in range(4):
        for b in range(4):
            assert c[a, b] == (FULL if b < a else PARTIAL if b == a else SKIP)


def test_tile_classes_golden_counts():
    """Regression values for the two prefill workloads, written by
    tests/golden/make_golden.py from the oracle only."""
    g = json.load(open(os.path.join(GOLDEN, "tile_counts.json")))
    for case in g["cases"]:
        pos = np.arange(case["S"])
        c = tile_classes(pos, pos, case["P"], case["W"], case["BM"], case["BN"])
        assert [int((c == k).sum()) for k in (SKIP, PARTIAL, FULL)] == case["skip_partial_full"]


# ------------------------------------------------------------- Reset PE ----
from oracle import attend_reset_pe, reset_positions  # noqa: E402
import oracle.prefix_sliding as _ops  # noqa: E402


def test_reset_positions_renumber_the_cache_in_order():
    for P, W in ((4, 8), (0, 5), (16, 32), (3, 1)):
        for p in range(0, 120):
            js, reset, rq = reset_positions(p, P, W)
            L = min(p + 1, P + W)
            assert len(js) == L
            assert np.array_equal(reset, np.arange(L))      # 0..L-1, cache order
            assert np.array_equal(reset[js < P], js[js < P])  # prefix keeps its positions
            assert rq == L - 1


def test_reset_pe_equals_continue_pe_before_any_eviction():
    seed, hq, hkv, d, theta = 23, 4, 2, 16, 1e4
    hist = synth.History(seed, 0, hkv, d)
    q = synth.bits_to_f64(synth.query_bits(seed, 0, np.arange(60), hq, d))
    for P, W in ((8, 32), (0, 60), (40, 10)):
        for p in range(0, 60):
            if p + 1 > P + W:
                continue
            o1, l1 = attend(q[p], p, P, W, hist.rows, theta)
            o2, l2 = attend_reset_pe(q[p], p, P, W, hist.rows, theta)
            assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _bruteforce_reset(q_raw, p, P, W, hist, theta):
    """Scalar Python, no rounding: every key rotated at its renumbered
    position (prefix 0..P-1, then the window oldest first), the query at the
    newest window entry's position; keys found by listing the two ranges."""
    keys = sorted(set(range(0, min(P, p + 1))) | set(range(max(0, p - W + 1), p + 1)))
    newpos = {j: r for r, j in enumerate(keys)}
    k_raw, v = hist(np.array(keys))
    hq, d = q_raw.shape
    hkv = k_raw.shape[1]

    def rot(vec, pos):
        out = [0.0] * d
        for i in range(d // 2):
            z = complex(vec[i], vec[i + d // 2]) * cmath.exp(1j * pos * theta ** (-2 * i / d))
            out[i], out[i + d // 2] = z.real, z.imag
        return out

    outs, lses = [], []
    for h in range(hq):
        qv = rot(list(q_raw[h]), newpos[p])
        ws = [math.exp(sum(a * b for a, b in zip(qv, rot(list(k_raw[n, h * hkv // hq]), newpos[j])))
                       / math.sqrt(d)) for n, j in enumerate(keys)]
        tot = sum(ws)
        outs.append([sum(ws[n] / tot * v[n, h * hkv // hq, t] for n in range(len(keys)))
                     for t in range(d)])
        lses.append(math.log(tot))
    return np.array(outs), np.array(lses)


def test_reset_pe_matches_explicit_renumbering_without_rounding(monkeypatch):
    """With the bf16 contract rounding switched off, the oracle's query-side
    rotation equals rotating every key at its renumbered position."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    seed, hq, hkv, d, theta = 24, 2, 1, 8, 1e4
    hist = synth.History(seed, 2, hkv, d)
    q = synth.bits_to_f64(synth.query_bits(seed, 2, np.arange(40), hq, d))
    for P, W in ((3, 5), (0, 4), (6, 1), (10, 30)):
        for p in range(0, 40, 3):
            o, l = _ops.attend_reset_pe(q[p], p, P, W, hist.rows, theta)
            ob, lb = _bruteforce_reset(q[p], p, P, W, hist.rows, theta)
            assert np.allclose(o, ob, atol=1e-12) and np.allclose(l, lb, atol=1e-12), (P, W, p)


def test_reset_pe_without_prefix_is_a_uniform_shift(monkeypatch):
    """P = 0: every key is a window key, renumbering shifts all positions by
    the same amount, so (without rounding) Reset PE equals Continue PE."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    seed, hq, hkv, d, theta = 25, 2, 1, 16, 1e4
    hist = synth.History(seed, 3, hkv, d)
    q = synth.bits_to_f64(synth.query_bits(seed, 3, np.arange(200), hq, d))
    for p in (50, 120, 199):
        o1, l1 = _ops.attend(q[p], p, 0, 17, hist.rows, theta)
        o2, l2 = _ops.attend_reset_pe(q[p], p, 0, 17, hist.rows, theta)
        assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


# ------------------------------------------------------------- backward ----
from oracle import attend_backward  # noqa: E402


def _bwd_inputs(seed, S, hq, hkv, d):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((S, hq, d))
    k = rng.standard_normal((S, hkv, d))
    v = rng.standard_normal((S, hkv, d))
    do = rng.standard_normal((S, hq, d))
    return q, k, v, do


@pytest.mark.parametrize("S,P,W", [(24, 5, 7), (20, 0, 4), (16, 16, 3), (19, 3, 40)])
def test_backward_matches_torch_autograd_of_sdpa(monkeypatch, S, P, W):
    """Rounding off: the hand-written gradients equal torch autograd through
    scaled_dot_product_attention with the explicit mask (float64), pulled back
    through the rotation by autograd as well."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    hq, hkv, d, theta = 4, 2, 8, 100.0
    q, k, v, do = _bwd_inputs(S * 7 + P, S, hq, hkv, d)
    dq, dk, dv, o, lse = _ops.attend_backward(q, k, v, do, P, W, theta)
    pos = torch.arange(S, dtype=torch.float64)
    inv = theta ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    ang = pos[:, None] * inv[None, :]
    c, s_ = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]

    def rot(x):  # half-split rotation written with torch ops, differentiable
        x1, x2 = x[..., : d // 2], x[..., d // 2:]
        return torch.cat([x1 * c - x2 * s_, x2 * c + x1 * s_], dim=-1)

    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    qh = rot(tq).permute(1, 0, 2)
    kh = rot(tk).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    vh = tv.permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    jj, pp = torch.meshgrid(torch.arange(S), torch.arange(S), indexing="xy")
    mask = (jj <= pp) & ((jj < P) | (jj > pp - W))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask)
    out.backward(torch.tensor(do).permute(1, 0, 2))
    assert np.allclose(o, out.detach().permute(1, 0, 2).numpy(), atol=1e-12)
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-10)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-10)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-10)


@pytest.mark.parametrize("S,c0,P,W", [(20, 5, 12, 6), (18, 37, 10, 5), (16, 3, 0, 4)])
def test_backward_at_offset_positions_matches_torch_autograd(monkeypatch, S, c0, P, W):
    """A chunk at positions c0 .. c0 + S - 1 with no earlier keys: rotations and
    the mask use absolute positions (prefix keys only where c0 + j < P)."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    hq, hkv, d, theta = 2, 1, 8, 100.0
    q, k, v, do = _bwd_inputs(S + 3 * c0, S, hq, hkv, d)
    positions = c0 + np.arange(S)
    dq, dk, dv, o, _ = _ops.attend_backward(q, k, v, do, P, W, theta, positions=positions)
    pos = torch.tensor(positions, dtype=torch.float64)
    inv = theta ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    ang = pos[:, None] * inv[None, :]
    c, s_ = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]

    def rot(x):
        x1, x2 = x[..., : d // 2], x[..., d // 2:]
        return torch.cat([x1 * c - x2 * s_, x2 * c + x1 * s_], dim=-1)

    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    qh = rot(tq).permute(1, 0, 2)
    kh = rot(tk).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    vh = tv.permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    jj, pp = torch.meshgrid(pos, pos, indexing="xy")
    mask = (jj <= pp) & ((jj < P) | (jj > pp - W))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask)
    out.backward(torch.tensor(do).permute(1, 0, 2))
    assert np.allclose(o, out.detach().permute(1, 0, 2).numpy(), atol=1e-12)
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-10)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-10)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-10)


def test_backward_matches_finite_differences(monkeypatch):
    """Rounding off: d(sum(dO * O))/dq, dk, dv by central differences."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    S, hq, hkv, d, P, W, theta = 9, 2, 1, 4, 2, 3, 50.0
    q, k, v, do = _bwd_inputs(3, S, hq, hkv, d)
    dq, dk, dv, _, _ = _ops.attend_backward(q, k, v, do, P, W, theta)

    def loss(qq, kk, vv):
        return float((_ops.attend_backward(qq, kk, vv, do, P, W, theta)[3] * do).sum())

    eps = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [q.copy(), k.copy(), v.copy()]
            minus = [q.copy(), k.copy(), v.copy()]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-6, (which, idx, fd, grad[idx])


def test_backward_forward_equals_attend():
    seed, S, hq, hkv, d, P, W, theta = 26, 30, 4, 2, 16, 6, 9, 1e4
    hist = synth.History(seed, 0, hkv, d)
    pos = np.arange(S)
    q = synth.bits_to_f64(synth.query_bits(seed, 0, pos, hq, d))
    k, v = hist.rows(pos)
    _, _, _, o, lse = attend_backward(q, k, v, np.zeros_like(q), P, W, theta)
    for p in range(S):
        o_ref, l_ref = attend(q[p], p, P, W, hist.rows, theta)
        assert np.allclose(o[p], o_ref, atol=1e-13) and np.allclose(lse[p], l_ref, atol=1e-13)


def _autograd_grads(q, k, v, do, P, W, theta, positions):
    """torch autograd of SDPA (float64) with the explicit mask, through the rotation."""
    S, hq, d = q.shape
    hkv = k.shape[1]
    pos = torch.tensor(positions, dtype=torch.float64)
    inv = theta ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    ang = pos[:, None] * inv[None, :]
    c, s_ = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]

    def rot(x):
        x1, x2 = x[..., : d // 2], x[..., d // 2:]
        return torch.cat([x1 * c - x2 * s_, x2 * c + x1 * s_], dim=-1)

    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    qh = rot(tq).permute(1, 0, 2)
    kh = rot(tk).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    vh = tv.permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    jj, pp = torch.meshgrid(pos, pos, indexing="xy")
    mask = (jj <= pp) & ((jj < P) | (jj > pp - W))
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask)
    out.backward(torch.tensor(do).permute(1, 0, 2))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("S,c0,P,W,hq,hkv", [(40, 0, 6, 9, 4, 2), (33, 0, 0, 5, 2, 2),
                                             (30, 17, 20, 6, 4, 1), (28, 0, 28, 4, 2, 1)])
def test_backward_at_selected_rows_matches_torch_autograd(monkeypatch, S, c0, P, W, hq, hkv):
    """Rounding off: dq at chosen query rows and dk, dv at chosen key rows (prefix
    keys, keys at the prefix / window edge, the last key) equal the same rows of
    torch autograd through SDPA with the explicit mask."""
    monkeypatch.setattr(_ops, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    d, theta = 8, 100.0
    q, k, v, do = _bwd_inputs(S * 5 + P + c0, S, hq, hkv, d)
    positions = c0 + np.arange(S)
    q_rows = [0, 1, P // 2, max(P - 1, 0), min(P, S - 1), S // 2, S - 1]
    k_rows = [0, max(P - 1, 0), min(P, S - 1), S - W, S - 2, S - 1]
    dq, dk, dv = _ops.attend_backward_at(q, k, v, do, P, W, theta, q_rows, k_rows,
                                         positions=positions)
    gq, gk, gv = _autograd_grads(q, k, v, do, P, W, theta, positions)
    assert np.allclose(dq, gq[q_rows], atol=1e-10)
    assert np.allclose(dk, gk[k_rows], atol=1e-10)
    assert np.allclose(dv, gv[k_rows], atol=1e-10)


def test_backward_at_rounds_like_backward():
    """With the bf16 rounding contract on, the selected rows equal the same rows of
    the whole-sequence gradients."""
    seed, S, hq, hkv, d, P, W, theta = 27, 36, 4, 2, 16, 5, 11, 1e4
    hist = synth.History(seed, 0, hkv, d)
    pos = np.arange(S)
    q = synth.bits_to_f64(synth.query_bits(seed, 0, pos, hq, d))
    k, v = hist.rows(pos)
    do = synth.bits_to_f64(synth.normal_bf16(seed, 5, 0, pos, hq, d))
    full = attend_backward(q, k, v, do, P, W, theta)
    rows = [0, 4, 5, 20, 35]
    dq, dk, dv = _ops.attend_backward_at(q, k, v, do, P, W, theta, rows, rows)
    assert np.allclose(dq, full[0][rows], atol=1e-12)
    assert np.allclose(dk, full[1][rows], atol=1e-12)
    assert np.allclose(dv, full[2][rows], atol=1e-12)
