"""The bounded-wait failure path, exercised without faulting anything (GPU).

With the library's test hook on, CTA 0 of the next kernels skips its first K/V
copy (no copy is issued, so nothing is left in flight) and the waits give up
after 1 ms: the call must set PS_DEV_TIMEOUT, let everything it did issue land,
release its memory and return.  The next normal call on the same stream must
then be correct.
"""
import contextlib

import numpy as np
import pytest
import torch

import synth
from oracle import attend

from _util import (append_runs, assert_attention_close, bf16_tensor_to_f64, bits_to_bf16_tensor,
                   live_runs, synth_source)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


@contextlib.contextmanager
def forced_timeout(ps, limit_ns=1_000_000):
    assert ps.lib.ps_test_force_wait_timeout(1, limit_ns) == 0
    try:
        yield
    finally:
        assert ps.lib.ps_test_force_wait_timeout(0, 0) == 0


def test_hook_arguments(ps):
    assert ps.lib.ps_test_force_wait_timeout(2, 10 ** 6) == 1
    assert ps.lib.ps_test_force_wait_timeout(1, 10) == 1          # below 1 us
    assert ps.lib.ps_test_force_wait_timeout(1, 10 ** 12) == 1    # above the default limit
    assert ps.lib.ps_test_force_wait_timeout(0, 0) == 0


def test_decode_wait_times_out_then_recovers(ps):
    # 4 sequences x 8 KV heads x ~270 tiles: every warp of the grid owns tiles
    seed, nseq, hq, hkv, D, W, theta = 51, 4, 16, 8, 128, 4096, 10000.0
    P, pos = [100, 7, 300, 64], [9000, 5000, 20000, 4300]
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta)
    append_runs(cache, {s: live_runs(pos[s], P[s], W) for s in range(nseq)},
                synth_source(seed, hkv, D))
    q = bits_to_bf16_tensor(np.concatenate(
        [synth.query_bits(seed, s, pos[s], hq, D) for s in range(nseq)]))
    tpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    with forced_timeout(ps):
        cache.decode(q, tpos)
        torch.cuda.synchronize()
    assert cache.check_status() == ps.PS_DEV_TIMEOUT
    cache.status.zero_()
    o, lse = cache.decode(q, tpos)
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for s in range(nseq):
        qs = synth.bits_to_f64(synth.query_bits(seed, s, pos[s], hq, D))[0]
        o_ref, l_ref = attend(qs, pos[s], P[s], W, synth.History(seed, s, hkv, D).rows, theta)
        assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), o_ref, l_ref,
                               f"after timeout, seq {s}")


@pytest.mark.parametrize("hq,hkv", [(4, 2), (2, 2)])   # the pair kernel, the single-head kernel
def test_prefill_wait_times_out_then_recovers(ps, hq, hkv):
    seed, B, S, D, P, W, theta = 52, 2, 300, 128, [37, 5], 100, 10000.0
    pos = np.arange(S)
    q = np.stack([synth.query_bits(seed, b, pos, hq, D) for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(pos) for b in range(B)]
    tq = bits_to_bf16_tensor(q)
    tk = bits_to_bf16_tensor(np.stack([x[0] for x in kv]))
    tv = bits_to_bf16_tensor(np.stack([x[1] for x in kv]))
    i32 = dict(dtype=torch.int32, device="cuda")
    qs, pl = torch.zeros(B, **i32), torch.tensor(P, **i32)
    status = torch.zeros(1, **i32)
    torch.cuda.synchronize()
    with forced_timeout(ps):
        ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
        torch.cuda.synchronize()
    assert int(status.item()) == ps.PS_DEV_TIMEOUT
    status.zero_()
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(B):
        hist = synth.History(seed, b, hkv, D)
        for r in (0, 36, 37, 100, 136, 137, 200, 299):
            o_ref, l_ref = attend(synth.bits_to_f64(q[b, r]), r, P[b], W, hist.rows, theta)
            assert_attention_close(bf16_tensor_to_f64(out[b, r]), lse[b, :, r].cpu().numpy(),
                                   o_ref, l_ref, f"after timeout, b={b} row={r}")


def test_backward_wait_times_out_then_recovers(ps):
    from oracle import attend_backward
    seed, B, S, hq, hkv, D, P, W, theta = 53, 1, 300, 4, 2, 128, [37], 100, 10000.0
    pos = np.arange(S)
    q = synth.query_bits(seed, 0, pos, hq, D)[None]
    k, v = synth.History(seed, 0, hkv, D).rows_bits(pos)
    do = synth.normal_bf16(seed, 5, 0, pos, hq, D)[None]
    tq, tk, tv, tdo = (bits_to_bf16_tensor(x) for x in (q, k[None], v[None], do))
    i32 = dict(dtype=torch.int32, device="cuda")
    qs, pl = torch.zeros(B, **i32), torch.tensor(P, **i32)
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    with forced_timeout(ps):
        ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta, status=status)
        torch.cuda.synchronize()
    assert int(status.item()) == ps.PS_DEV_TIMEOUT
    status.zero_()
    dq, dk, dv = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    refs = attend_backward(synth.bits_to_f64(q[0]), synth.bits_to_f64(k), synth.bits_to_f64(v),
                           synth.bits_to_f64(do[0]), P[0], W, theta)[:3]
    for got, ref, name in zip((dq, dk, dv), refs, ("dq", "dk", "dv")):
        g = got[0].double().cpu().numpy()
        for h in range(ref.shape[1]):
            scale = float(np.abs(ref[:, h]).max())
            assert np.abs(g[:, h] - ref[:, h]).max() <= 2e-2 * scale, f"{name} head {h}"
