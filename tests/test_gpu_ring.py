"""Ring-slot mapping and ps_kv_append against the oracle (GPU, bit-exact slots)."""
import numpy as np
import pytest
import torch

import synth
from oracle import RingSim, ring_slot, rope, round_bf16

from _util import append_runs, bf16_tensor_to_f64, bits_to_bf16_tensor, synth_source

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def test_ring_slots_bit_exact(ps):
    rng = np.random.default_rng(0)
    n = 200000
    W = 4096
    pos = rng.integers(0, 2**31 - 1, n).astype(np.int32)
    pos[:1000] = np.arange(1000)
    P = rng.integers(0, 600, n).astype(np.int32)
    got = ps.ring_slots(torch.from_numpy(pos).cuda(), torch.from_numpy(P).cuda(), W).cpu().numpy()
    want = np.array([ring_slot(int(a), int(b), W) for a, b in zip(pos, P)], dtype=np.int32)
    assert np.array_equal(got, want)
    for W2 in (1, 7, 8192):
        got = ps.ring_slots(torch.from_numpy(pos).cuda(), torch.from_numpy(P).cuda(), W2).cpu().numpy()
        want = np.array([ring_slot(int(a), int(b), W2) for a, b in zip(pos[:5000], P[:5000])])
        assert np.array_equal(got[:5000], want)


def _check_ring_contents(cache, seq, sim, hist, theta, D):
    """Pool rows of `seq` vs the oracle's ring simulation: V exact, K within
    one bf16 ulp of the oracle's rotated-and-rounded key, flips rare."""
    rows = cache.rows_of(seq).to(cache.k_pool.device)
    kp = bf16_tensor_to_f64(cache.k_pool[rows])
    vp = bf16_tensor_to_f64(cache.v_pool[rows])
    held = sim.slots
    slots = np.nonzero(held >= 0)[0]
    kraw, vraw = hist.rows(held[slots])
    kref = round_bf16(rope(kraw, held[slots], theta))
    assert np.array_equal(vp[slots], vraw)
    diff = np.abs(kp[slots] - kref)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(kref), 1e-30))) - 7)
    # The kernel rotates in fp32: its absolute error is about 1e-7 times the
    # norm of the rotated pair (x_i, x_{i+D/2}), which exceeds one bf16 ulp of
    # the result only where the two terms of the rotation nearly cancel.
    half = D // 2
    pair = np.sqrt(kraw[..., :half] ** 2 + kraw[..., half:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    assert np.all(diff <= ulp * 1.0001 + 2e-6 * pair), "rotated key off by more than one bf16 ulp"
    flips = np.count_nonzero(diff)
    assert flips <= max(2, 1e-3 * diff.size), f"{flips} of {diff.size} keys differ by one ulp"
    # untouched slots stay zero
    rest = np.nonzero(held < 0)[0]
    assert not np.any(kp[rest]) and not np.any(vp[rest])


@pytest.mark.parametrize("P,W,D,steps,chunk", [(16, 32, 64, 300, 1), (16, 32, 64, 300, 37),
                                               (0, 5, 128, 77, 200), (100, 4096, 128, 9000, 3000),
                                               (7, 1, 64, 40, 9)])
def test_append_matches_ring_simulation(ps, P, W, D, steps, chunk):
    seed, hkv, theta = 5, 2, 10000.0
    cache = ps.RingCache(1, hkv, D, W, [P], rope_theta=theta)
    hist = synth.History(seed, 0, hkv, D)
    sim = RingSim(P, W)
    p = 0
    while p < steps:
        n = min(chunk, steps - p)
        append_runs(cache, {0: [(p, n)]}, synth_source(seed, hkv, D))
        for x in range(p, p + n):
            sim.append(x)
        p += n
        sim.check(p - 1)
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    _check_ring_contents(cache, 0, sim, hist, theta, D)


@pytest.mark.parametrize("block_size", [16, 48])
def test_append_paged_matches_ring_simulation(ps, block_size):
    """Paged cache: the same appends land in the blocks a shuffled block table
    names; read back through the table they equal the ring simulation."""
    seed, hkv, D, W, theta = 6, 2, 128, 100, 10000.0
    P = [7, 30, 0]
    ends = [900, 64, 350]
    nseq = len(P)
    probe = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, block_size=block_size, device="cpu")
    nblocks = nseq * probe.blocks_per_seq
    order = np.random.default_rng(1).permutation(nblocks)
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, block_size=block_size,
                         block_order=order)
    runs = {s: [(0, ends[s] // 2), (ends[s] // 2, ends[s] - ends[s] // 2)] for s in range(nseq)}
    append_runs(cache, runs, synth_source(seed, hkv, D))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for s in range(nseq):
        sim = RingSim(P[s], W)
        for x in range(ends[s]):
            sim.append(x)
        _check_ring_contents(cache, s, sim, synth.History(seed, s, hkv, D), theta, D)


def test_append_many_sequences_one_call(ps):
    seed, hkv, D, W, theta = 9, 8, 128, 64, 5e5
    P = [0, 3, 64, 17]
    ends = [10, 500, 129, 1000]
    cache = ps.RingCache(4, hkv, D, W, P, rope_theta=theta)
    runs = {s: [(0, ends[s])] for s in range(4)}
    append_runs(cache, runs, synth_source(seed, hkv, D))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for s in range(4):
        sim = RingSim(P[s], W)
        for x in range(ends[s]):
            sim.append(x)
        _check_ring_contents(cache, s, sim, synth.History(seed, s, hkv, D), theta, D)


def test_append_device_checks_flag_bad_input(ps):
    cache = ps.RingCache(2, 1, 64, 8, [4, 4], prefix_max=4)
    k = torch.zeros(2, 1, 64, dtype=torch.bfloat16, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    # sequence index out of range -> PS_DEV_BAD_SEQ, nothing written
    cache.append(torch.tensor([5], **i32), torch.tensor([0], **i32), torch.tensor([0, 2], **i32), k, k)
    torch.cuda.synchronize()
    assert cache.check_status() & ps.PS_DEV_BAD_SEQ
    cache.status.zero_()
    # negative position -> PS_DEV_BAD_POS
    cache.append(torch.tensor([1], **i32), torch.tensor([-3], **i32), torch.tensor([0, 2], **i32), k, k)
    torch.cuda.synchronize()
    assert cache.check_status() & ps.PS_DEV_BAD_POS
    assert not torch.any(cache.k_pool.float() != 0)
