"""ps_decode_noalloc: the decode entry point for callers that cannot allocate
device memory when they decode (no allocator of their own, an allocator that
is locked or shutting down, or a budget that forbids growth during
generation).  It keeps its scratch in a fixed array inside the library.

Checked through the C ABI against ps_decode with a caller-allocated workspace,
on two calls in a row (the second call reuses the scratch the first one left
behind).  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

from _util import (append_runs, assert_attention_close, bf16_tensor_to_f64, bits_to_bf16_tensor,
                   live_runs, synth_source)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def _noalloc(ps, cache, q, pos, scale):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = ps.lib.ps_decode_noalloc(ctypes.byref(cache.desc), ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(pos.data_ptr()), q.shape[1],
                                    ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(lse.data_ptr()), stream)
    ps.check(code, "ps_decode_noalloc")
    return out, lse


def test_noalloc_decode_matches_workspace_decode_twice(ps):
    seed, hq, hkv, D, W, theta = 41, 16, 8, 128, 64, 10000.0
    P = [5, 0, 100, 37]
    pos0 = [300, 70, 120, 3000]
    nseq = len(P)
    scale = 1.0 / np.sqrt(D)
    cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta)
    append_runs(cache, {s: live_runs(pos0[s] - 1, P[s], W) for s in range(nseq)},
                synth_source(seed, hkv, D))
    for step in range(2):
        pos_host = [p + step for p in pos0]
        k, v = zip(*(synth.History(seed, s, hkv, D).rows_bits([pos_host[s]]) for s in range(nseq)))
        pos = torch.tensor(pos_host, dtype=torch.int32, device="cuda")
        cache.append_tokens(pos, bits_to_bf16_tensor(np.concatenate(k)),
                            bits_to_bf16_tensor(np.concatenate(v)))
        q = bits_to_bf16_tensor(np.concatenate(
            [synth.query_bits(seed, s, pos_host[s], hq, D) for s in range(nseq)]))
        o_ref, lse_ref = cache.decode(q, pos, scale=scale)
        o_na, lse_na = _noalloc(ps, cache, q, pos, scale)
        torch.cuda.synchronize()
        assert cache.check_status() == 0
        for s in range(nseq):
            assert_attention_close(bf16_tensor_to_f64(o_na[s]), lse_na[s].cpu().numpy(),
                                   bf16_tensor_to_f64(o_ref[s]), lse_ref[s].cpu().numpy().astype(np.float64),
                                   f"call {step + 1}, seq {s}")


def test_noalloc_scratch_left_by_a_different_layout(ps):
    """The scratch keeps whatever the previous call wrote.  A large call (many
    sequences, one of them refused by the device checks so that it owns no
    tiles) leaves its tile counts, segment bounds and records behind; the next,
    small call (fewer tiles than warps, so each warp owns at most one tile) must
    not read any of them.  Both calls are compared with ps_decode on a fresh
    workspace and with the oracle."""
    from oracle import attend
    seed, hq, hkv, D, W, theta = 43, 16, 8, 128, 256, 10000.0
    scale = 1.0 / np.sqrt(D)

    def run(nseq, P, pos, bad=None):
        cache = ps.RingCache(nseq, hkv, D, W, P, rope_theta=theta, prefix_max=max(P))
        append_runs(cache, {s: live_runs(pos[s], P[s], W) for s in range(nseq)},
                    synth_source(seed, hkv, D))
        if bad is not None:
            cache.prefix_len[bad] = 10 ** 6  # above prefix_max: sequence refused, no tiles
        q = bits_to_bf16_tensor(np.concatenate(
            [synth.query_bits(seed, s, pos[s], hq, D) for s in range(nseq)]))
        tpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
        ws = torch.empty(ps.decode_workspace_size(nseq, hq, hkv, D), dtype=torch.uint8,
                         device="cuda")
        o_ws, l_ws = cache.decode(q, tpos, scale=scale, workspace=ws)
        o_na, l_na = _noalloc(ps, cache, q, tpos, scale)
        torch.cuda.synchronize()
        flags = cache.check_status()
        assert flags == (ps.PS_DEV_BAD_PREFIX if bad is not None else 0)
        for s in range(nseq):
            if s == bad:
                assert torch.all(o_na[s].float() == 0) and torch.all(torch.isinf(l_na[s]))
                continue
            assert_attention_close(bf16_tensor_to_f64(o_na[s]), l_na[s].cpu().numpy(),
                                   bf16_tensor_to_f64(o_ws[s]), l_ws[s].cpu().numpy().astype(np.float64),
                                   f"nseq {nseq}, seq {s} vs ps_decode")
            if s < 6:
                qs = synth.bits_to_f64(synth.query_bits(seed, s, pos[s], hq, D))[0]
                o_ref, l_ref = attend(qs, pos[s], P[s], W, synth.History(seed, s, hkv, D).rows, theta)
                assert_attention_close(bf16_tensor_to_f64(o_na[s]), l_na[s].cpu().numpy(), o_ref,
                                       l_ref, f"nseq {nseq}, seq {s} vs oracle")

    rng = np.random.default_rng(4)
    n_big = 96
    P_big = rng.integers(0, 64, n_big).tolist()
    pos_big = rng.integers(300, 5000, n_big).tolist()
    run(n_big, P_big, pos_big, bad=5)                    # many tiles, one sequence without any
    run(2, [3, 0], [20, 40])                             # 2 x 8 heads x 3 tiles: far fewer than warps


def test_noalloc_rejects_shapes_beyond_its_scratch(ps):
    # 2,048 sequences x 8 KV heads need far more than the 4 MiB of fixed scratch;
    # the call must refuse before touching any pointer it was given.
    cache = ps.RingCache(1, 8, 128, 16, [0])
    desc = ps.CacheDesc.from_buffer_copy(cache.desc)
    desc.nseq = 2048
    q = torch.zeros(1, 16, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = ps.lib.ps_decode_noalloc(ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(pos.data_ptr()), 16, ctypes.c_float(0.1),
                                    ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(pos.data_ptr()),
                                    None)
    assert code == 4  # PS_ERR_WORKSPACE
