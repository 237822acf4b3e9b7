"""ps_kv_append + ps_decode against the float64 oracle, which attends from the
full, never-evicted history (GPU)."""
import numpy as np
import pytest
import torch

import synth
from oracle import attend, attend_reset_pe

from _util import (append_runs, assert_attention_close, bf16_tensor_to_f64, bits_to_bf16_tensor,
                   live_runs, lse_tol_stress, random_source, synth_source)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def _oracle_rows(seed, seqs, pos, P, W, hq, hkv, D, theta, qscale_log2=0):
    out = {}
    for s in seqs:
        q = synth.bits_to_f64(synth.query_bits(seed, s, pos[s], hq, D, qscale_log2))[0]
        out[s] = attend(q, int(pos[s]), int(P[s]), W, synth.History(seed, s, hkv, D).rows, theta)
    return out


def _queries(seed, nseq, pos, hq, D, qscale_log2=0):
    bits = np.concatenate([synth.query_bits(seed, s, pos[s], hq, D, qscale_log2) for s in range(nseq)])
    return bits_to_bf16_tensor(bits)


def _step_decode(ps, cache, seed, p, hq, hkv, D):
    """Decode step of one sequence: append token p, then attend with q at p."""
    k, v = synth.History(seed, 0, hkv, D).rows_bits([p])
    pos = torch.tensor([p], dtype=torch.int32, device="cuda")
    cache.append_tokens(pos, bits_to_bf16_tensor(k), bits_to_bf16_tensor(v))
    q = bits_to_bf16_tensor(synth.query_bits(seed, 0, p, hq, D))
    return cache.decode(q, pos)


def test_tiny_decode_240_steps_with_evictions(ps):
    """Batch 1, 2 query heads / 1 KV head, D=64, P=16, W=32; the 16-token
    prefix goes in as one chunk, then 240 decode steps (positions 16..255,
    208 evictions), each checked against the full-history oracle."""
    seed, hq, hkv, D, P, W, theta = 1, 2, 1, 64, 16, 32, 10000.0
    cache = ps.RingCache(1, hkv, D, W, [P], rope_theta=theta)
    append_runs(cache, {0: [(0, P)]}, synth_source(seed, hkv, D))
    hist = synth.History(seed, 0, hkv, D)
    for p in range(P, 256):
        o, lse = _step_decode(ps, cache, seed, p, hq, hkv, D)
        q = synth.bits_to_f64(synth.query_bits(seed, 0, p, hq, D))[0]
        o_ref, lse_ref = attend(q, p, P, W, hist.rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o[0]), lse[0].cpu().numpy(), o_ref, lse_ref, f"p={p}")
    assert cache.check_status() == 0


def test_decode_soak_4352_steps(ps):
    """Same shape for 4,352 steps (4,320 evictions); every step checked."""
    seed, hq, hkv, D, P, W, theta = 2, 2, 1, 64, 16, 32, 10000.0
    cache = ps.RingCache(1, hkv, D, W, [P], rope_theta=theta)
    hist = synth.History(seed, 0, hkv, D)
    for p in range(0, 4352):
        o, lse = _step_decode(ps, cache, seed, p, hq, hkv, D)
        q = synth.bits_to_f64(synth.query_bits(seed, 0, p, hq, D))[0]
        o_ref, lse_ref = attend(q, p, P, W, hist.rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o[0]), lse[0].cpu().numpy(), o_ref, lse_ref, f"p={p}")
    assert cache.check_status() == 0


CASES = [
    # nseq, Hq, Hkv, D, P per seq, W, pos per seq, q scale (log2)
    (3, 16, 8, 128, [100, 0, 7], 64, [50, 1000, 170], 0),
    (2, 4, 4, 128, [5, 300], 16, [4, 299], 0),          # G=1; p < P; p+1 = P
    (2, 8, 2, 64, [0, 33], 1, [0, 5000], 0),             # G=4; W=1; p = 0
    (2, 8, 1, 128, [64, 64], 200, [263, 264], 0),        # G=8; L = P+W-? around the fill point
    (4, 16, 8, 128, [512, 64, 300, 1], 4096, [131072, 4159, 4395, 262143], 0),
    (2, 16, 8, 128, [100, 100], 4096, [10000, 4196], 2),  # q x 4: sharper softmax
    (1, 2, 1, 64, [16], 32, [16], 0),
]


@pytest.mark.parametrize("nseq,hq,hkv,D,P,W,pos,qs", CASES)
def test_decode_shapes_and_edges(ps, nseq, hq, hkv, D, P, W, pos, qs):
    seed, theta = 7, 10000.0
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta)
    runs = {s: live_runs(pos[s], P[s], W) for s in range(nseq)}
    append_runs(cache, runs, synth_source(seed, hkv, D))
    q = _queries(seed, nseq, pos, hq, D, qs)
    o, lse = cache.decode(q, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    ref = _oracle_rows(seed, range(nseq), pos, P, W, hq, hkv, D, theta, qs)
    for s in range(nseq):
        assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), *ref[s], f"seq {s}",
                               lse_abs=lse_tol_stress(qs))


PAGED_CASES = [
    # nseq, Hq, Hkv, D, P per seq, W, pos per seq, block size
    (3, 16, 8, 128, [100, 0, 7], 64, [50, 1000, 170], 16),
    (4, 16, 8, 128, [512, 64, 300, 1], 4096, [131072, 4159, 4395, 262143], 64),
    (2, 8, 2, 64, [0, 33], 1, [0, 5000], 32),
]


@pytest.mark.parametrize("nseq,hq,hkv,D,P,W,pos,bs", PAGED_CASES)
def test_decode_paged_cache(ps, nseq, hq, hkv, D, P, W, pos, bs):
    """Paged cache behind a shuffled block table: same results as the oracle."""
    seed, theta = 12, 10000.0
    probe = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, block_size=bs, device="cpu")
    order = np.random.default_rng(3).permutation(nseq * probe.blocks_per_seq)
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, block_size=bs, block_order=order)
    append_runs(cache, {s: live_runs(pos[s], P[s], W) for s in range(nseq)},
                synth_source(seed, hkv, D))
    q = _queries(seed, nseq, pos, hq, D)
    o, lse = cache.decode(q, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    ref = _oracle_rows(seed, range(nseq), pos, P, W, hq, hkv, D, theta)
    for s in range(nseq):
        assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), *ref[s], f"seq {s}")


def test_decode_paged_block_outside_pool_is_flagged(ps):
    """A block id outside the pool is reported, and nothing outside the pool is read."""
    seed, hq, hkv, D, W = 13, 4, 2, 128, 32
    cache = ps.RingCache(2, hkv, D, W, [4, 4], rope_theta=1e4, block_size=16)
    append_runs(cache, {s: live_runs(40, 4, W) for s in range(2)}, synth_source(seed, hkv, D))
    cache.block_table[1, 1] = 10 ** 6
    q = _queries(seed, 2, [40, 40], hq, D)
    o, lse = cache.decode(q, torch.tensor([40, 40], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() & ps.PS_DEV_BAD_SLOT
    ref = _oracle_rows(seed, [0], [40, 40], [4, 4], W, hq, hkv, D, 1e4)
    assert_attention_close(bf16_tensor_to_f64(o[0]), lse[0].cpu().numpy(), *ref[0], "seq 0")


def _full_size_case(ps, seed, nseq, pos, P, W, sampled):
    hq, hkv, D, theta = 16, 8, 128, 10000.0
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, prefix_max=512)
    syn = synth_source(seed, hkv, D)
    rnd = random_source(seed + 1000, hkv, D)
    runs = {s: live_runs(int(pos[s]), int(P[s]), W) for s in range(nseq)}
    append_runs(cache, {s: r for s, r in runs.items() if s in sampled}, syn)
    append_runs(cache, {s: r for s, r in runs.items() if s not in sampled}, rnd)
    qbits = np.concatenate([synth.query_bits(seed, s, int(pos[s]), hq, D) for s in range(nseq)])
    q = bits_to_bf16_tensor(qbits)
    o, lse = cache.decode(q, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    ref = _oracle_rows(seed, sampled, pos, P, W, hq, hkv, D, theta)
    for s in sampled:
        assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), *ref[s], f"seq {s}")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return cache


def test_steady_decode_full_size_sampled(ps):
    """64 sequences at position 131,072, P uniform in 64..512, W = 4,096,
    16/8 heads, D = 128, in the launch configuration the benchmark times;
    4 sequences checked against the oracle."""
    seed, nseq, W = 3, 64, 4096
    P = synth.uniform_int(seed, 10, nseq, 64, 512)
    pos = np.full(nseq, 131072)
    _full_size_case(ps, seed, nseq, pos, P, W, sampled=[0, 17, 42, 63])


def test_ragged_decode_full_size_sampled(ps):
    """256 sequences, positions uniform in [1024, 262144], P in 64..512,
    W = 8,192; the sample includes sequences still in the causal regime."""
    seed, nseq, W = 4, 256, 8192
    P = synth.uniform_int(seed, 10, nseq, 64, 512)
    pos = synth.uniform_int(seed, 11, nseq, 1024, 262143)
    causal = [int(s) for s in np.nonzero(pos + 1 < P + W)[0]][:3]
    sampled = sorted(set(causal + [0, 100, 255]))
    assert causal, "the recipe should put a few sequences below P + W"
    _full_size_case(ps, seed, nseq, pos, P, W, sampled)


def test_decode_flags_bad_prefix_and_keeps_others(ps):
    seed, hq, hkv, D, W = 8, 4, 2, 128, 16
    P = [3, 3]
    cache = ps.RingCache(2, hkv, D, W, P, rope_theta=1e4)
    pos = [40, 41]
    append_runs(cache, {s: live_runs(pos[s], P[s], W) for s in range(2)}, synth_source(seed, hkv, D))
    cache.prefix_len[1] = 99  # above prefix_max: the kernel must refuse sequence 1
    q = _queries(seed, 2, pos, hq, D)
    o, lse = cache.decode(q, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() & ps.PS_DEV_BAD_PREFIX
    assert torch.all(o[1].float() == 0) and torch.all(torch.isinf(lse[1]))
    ref = _oracle_rows(seed, [0], pos, P, W, hq, hkv, D, 1e4)
    assert_attention_close(bf16_tensor_to_f64(o[0]), lse[0].cpu().numpy(), *ref[0], "seq 0")


# ---------------------------------------------------------------- Reset PE --
def test_tiny_decode_reset_pe_240_steps(ps):
    """Reset PE (cache renumbered in order each step): the tiny workload,
    every step against the full-history oracle of the renumbered positions."""
    seed, hq, hkv, D, P, W, theta = 1, 2, 1, 64, 16, 32, 10000.0
    cache = ps.RingCache(1, hkv, D, W, [P], rope_theta=theta, pe_mode=ps.PS_PE_RESET)
    append_runs(cache, {0: [(0, P)]}, synth_source(seed, hkv, D))
    hist = synth.History(seed, 0, hkv, D)
    for p in range(P, 256):
        o, lse = _step_decode(ps, cache, seed, p, hq, hkv, D)
        q = synth.bits_to_f64(synth.query_bits(seed, 0, p, hq, D))[0]
        o_ref, lse_ref = attend_reset_pe(q, p, P, W, hist.rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o[0]), lse[0].cpu().numpy(), o_ref, lse_ref, f"p={p}")
    assert cache.check_status() == 0


@pytest.mark.parametrize("nseq,hq,hkv,D,P,W,pos", [
    (4, 16, 8, 128, [100, 0, 7, 37], 64, [50, 1000, 170, 100]),       # below / above the fill point
    (3, 16, 8, 128, [100, 512, 64], 4096, [10000, 131072, 4200]),      # prefix / window boundary mid-tile
    (2, 8, 1, 128, [5, 20], 16, [300, 45]),                            # G = 8
])
def test_decode_reset_pe_shapes(ps, nseq, hq, hkv, D, P, W, pos):
    seed, theta = 14, 10000.0
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, pe_mode=ps.PS_PE_RESET)
    append_runs(cache, {s: live_runs(pos[s], P[s], W) for s in range(nseq)}, synth_source(seed, hkv, D))
    q = _queries(seed, nseq, pos, hq, D)
    o, lse = cache.decode(q, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for s in range(nseq):
        qs = synth.bits_to_f64(synth.query_bits(seed, s, pos[s], hq, D))[0]
        o_ref, l_ref = attend_reset_pe(qs, pos[s], P[s], W, synth.History(seed, s, hkv, D).rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), o_ref, l_ref, f"seq {s}")


def test_decode_graph_replays_the_eager_step(ps):
    """DecodeGraph (append + decode captured once by the library, then launched per
    step, alternately on inputs filled on the device and through one native call
    that copies packed host blocks in and out) gives the same bits as the eager
    calls on an identical cache, and stays within the oracle's tolerance, across
    steps that evict."""
    seed, nseq, hq, hkv, D, W, theta = 17, 3, 4, 2, 128, 64, 10000.0
    P = np.array([5, 40, 0])
    pos0 = np.array([100, 70, 300])
    caches = []
    for _ in range(2):
        c = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta)
        runs = {s: live_runs(int(pos0[s]) - 1, int(P[s]), W) for s in range(nseq)}
        append_runs(c, runs, synth_source(seed, hkv, D))
        caches.append(c)
    torch.cuda.synchronize()
    eager, graphed = caches
    g = ps.DecodeGraph(graphed, hq)
    for step in range(20):
        pos = pos0 + step
        kv = [synth.History(seed, s, hkv, D).rows_bits([int(pos[s])]) for s in range(nseq)]
        k = bits_to_bf16_tensor(np.concatenate([x[0] for x in kv]))
        v = bits_to_bf16_tensor(np.concatenate([x[1] for x in kv]))
        q = _queries(seed, nseq, pos, hq, D)
        tpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
        eager.append_tokens(tpos, k, v)
        o_e, l_e = eager.decode(q, tpos)
        if step % 2 == 0:  # inputs filled on the device, graph launched alone
            g.q.copy_(q)
            g.k.copy_(k)
            g.v.copy_(v)
            g.pos.copy_(tpos)
            g.replay()
            torch.cuda.synchronize()
            o_g, l_g = g.out, g.lse
        else:  # one native call: packed host block in, step, packed results out
            hin = torch.zeros(g.inp.numel(), dtype=torch.uint8)
            hres = torch.zeros(g.res.numel(), dtype=torch.uint8)
            if step % 4 == 1:  # page-locked, the serving case; else pageable
                hin, hres = hin.pin_memory(), hres.pin_memory()
            for name, t in (("q", q), ("k", k), ("v", v), ("pos", tpos)):
                o, nb = g.in_layout[name]
                hin[o:o + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            g.step(hin, hres)
            o, nb = g.res_layout["out"]
            o_g = hres[o:o + nb].view(torch.bfloat16).view(o_e.shape).cuda()
            o, nb = g.res_layout["lse"]
            l_g = hres[o:o + nb].view(torch.float32).view(l_e.shape).cuda()
        assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e), step
    ref = _oracle_rows(seed, range(nseq), pos, P, W, hq, hkv, D, theta)
    for s in range(nseq):
        assert_attention_close(g.out[s].float().cpu().numpy(), g.lse[s].cpu().numpy(), *ref[s])
    assert eager.check_status() == 0 and graphed.check_status() == 0
    g.close()
    g.close()  # a second close is a no-op


# ------------------------------------------------------------- fused append --
@pytest.mark.parametrize("nseq,hq,hkv,D,P,W,pos0,pe,bs", [
    (3, 16, 8, 128, [100, 0, 7], 64, [50, 1000, 170], 0, None),     # causal / evicting mixes
    (2, 8, 2, 64, [0, 33], 16, [0, 5000], 0, None),                 # D 64, first token, W 16
    (4, 16, 8, 128, [512, 64, 300, 1], 4096, [131072, 4159, 4395, 262143], 1, None),  # Reset PE
    (3, 16, 8, 128, [100, 0, 7], 64, [50, 1000, 170], 0, 16),       # paged
])
def test_decode_append_equals_append_then_decode(ps, nseq, hq, hkv, D, P, W, pos0, pe, bs):
    """ps_decode_append over 40 steps (each evicting) leaves the same cache bits and
    returns the same out / lse bits as ps_kv_append followed by ps_decode, and
    matches the oracle."""
    seed, theta = 18, 10000.0
    pos0 = np.array(pos0)
    caches = []
    for _ in range(2):
        kw = dict(rope_theta=theta, pe_mode=pe)
        if bs:
            probe = ps.RingCache(nseq, hkv, D, W, P, block_size=bs, device="cpu", **kw)
            kw.update(block_size=bs,
                      block_order=np.random.default_rng(7).permutation(nseq * probe.blocks_per_seq))
        c = ps.RingCache(nseq, hkv, D, W, P, **kw)
        append_runs(c, {s: live_runs(int(pos0[s]) - 1, P[s], W) for s in range(nseq)
                        if pos0[s] > 0}, synth_source(seed, hkv, D))
        caches.append(c)
    sep, fused = caches
    for step in range(40):
        pos = pos0 + step
        kv = [synth.History(seed, s, hkv, D).rows_bits([int(pos[s])]) for s in range(nseq)]
        k = bits_to_bf16_tensor(np.concatenate([x[0] for x in kv]))
        v = bits_to_bf16_tensor(np.concatenate([x[1] for x in kv]))
        q = _queries(seed, nseq, pos, hq, D)
        tpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
        sep.append_tokens(tpos, k, v)
        o_a, l_a = sep.decode(q, tpos)
        o_b, l_b = fused.decode_append(q, k, v, tpos)
        torch.cuda.synchronize()
        assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b), step
    assert torch.equal(sep.k_pool, fused.k_pool) and torch.equal(sep.v_pool, fused.v_pool)
    assert sep.check_status() == 0 and fused.check_status() == 0
    ref = attend_reset_pe if pe else attend
    for s in range(nseq):
        qs = synth.bits_to_f64(synth.query_bits(seed, s, int(pos[s]), hq, D))[0]
        o_ref, l_ref = ref(qs, int(pos[s]), P[s], W, synth.History(seed, s, hkv, D).rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o_b[s]), l_b[s].cpu().numpy(), o_ref, l_ref,
                               f"seq {s}")


def test_decode_with_per_sequence_slot_bases(ps):
    """Full-history caches whose sequences stop at different positions, packed with
    per-sequence pool bases: each sequence's reservation (capacity rows) overlaps the
    next sequences', but the rows it fills do not.  Decode over a few appended steps
    matches the oracle, and the rows past each sequence's filled slots are untouched."""
    seed, hq, hkv, D, theta, steps = 23, 4, 2, 128, 10000.0, 3
    pos0 = np.array([50, 300, 130])
    nseq = len(pos0)
    W = int(pos0.max()) + steps + 1          # no eviction: every position stays
    P = np.zeros(nseq, dtype=np.int64)
    used = pos0 + steps                      # slots each sequence fills
    base = np.concatenate([[0], np.cumsum(used)[:-1]])
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, slot_base=base.tolist())
    assert cache.k_pool.shape[0] == int(base.max()) + W
    append_runs(cache, {s: [(0, int(pos0[s]))] for s in range(nseq)}, synth_source(seed, hkv, D))
    for step in range(steps):
        pos = pos0 + step
        kv = [synth.History(seed, s, hkv, D).rows_bits([int(pos[s])]) for s in range(nseq)]
        k = bits_to_bf16_tensor(np.concatenate([x[0] for x in kv]))
        v = bits_to_bf16_tensor(np.concatenate([x[1] for x in kv]))
        tpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
        o, lse = cache.decode_append(_queries(seed, nseq, pos, hq, D), k, v, tpos)
        torch.cuda.synchronize()
        assert cache.check_status() == 0
        ref = _oracle_rows(seed, range(nseq), pos, P, W, hq, hkv, D, theta)
        for s in range(nseq):
            assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), *ref[s],
                                   f"step {step} seq {s}")
    # the last sequence's tail of its reservation was never written (zero-initialised)
    last = int(base[-1] + used[-1])
    assert torch.count_nonzero(cache.k_pool[last:]).item() == 0
