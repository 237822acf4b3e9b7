"""A whole serving flow through the public binding, as the README shows it: prompt
prefill, the prompt's K/V appended to the ring (longer than the window, so only
the prefix and the last W positions stay), decode steps that append and attend in
one call, and a step through the host-buffer executor -- every output against the
oracle's attention over the full, never-evicted history."""
import numpy as np
import pytest
import torch

import synth
from oracle import attend

from _util import assert_attention_close, bf16_tensor_to_f64, bits_to_bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def test_prefill_append_decode_and_executor(ps):
    seed, nseq, S, hq, hkv, D, W, theta = 29, 2, 300, 4, 2, 128, 128, 10000.0
    Pl = [37, 100]
    i32 = dict(dtype=torch.int32, device="cuda")
    hist = [synth.History(seed, s, hkv, D) for s in range(nseq)]

    def q_at(pos):  # raw queries [nseq, hq, D] at one position per sequence
        return np.concatenate([synth.query_bits(seed, s, [int(pos[s])], hq, D) for s in range(nseq)])

    def kv_at(pos):
        kv = [hist[s].rows_bits([int(pos[s])]) for s in range(nseq)]
        return np.concatenate([x[0] for x in kv]), np.concatenate([x[1] for x in kv])

    def check(o, lse, pos, what):
        for s in range(nseq):
            qs = synth.bits_to_f64(synth.query_bits(seed, s, [int(pos[s])], hq, D))[0]
            o_ref, l_ref = attend(qs, int(pos[s]), Pl[s], W, hist[s].rows, theta)
            assert_attention_close(bf16_tensor_to_f64(o[s]), lse[s].cpu().numpy(), o_ref, l_ref,
                                   f"{what} seq {s}")

    # prompt: positions 0 .. S-1 of each sequence
    prompt = np.arange(S)
    q = np.stack([synth.query_bits(seed, s, prompt, hq, D) for s in range(nseq)])
    kv = [hist[s].rows_bits(prompt) for s in range(nseq)]
    k = bits_to_bf16_tensor(np.stack([x[0] for x in kv]))
    v = bits_to_bf16_tensor(np.stack([x[1] for x in kv]))
    q_start = torch.zeros(nseq, **i32)
    P = torch.tensor(Pl, **i32)
    out, lse = ps.prefill(bits_to_bf16_tensor(q), k, v, q_start, P, W, rope_theta=theta)
    torch.cuda.synchronize()
    for r in (0, Pl[0], W + 7, S - 1):  # rows before, at and past the window's first fill
        check(out[:, r], lse[:, :, r], [r] * nseq, f"prefill row {r}")

    cache = ps.RingCache(nseq, hkv, D, W, Pl, rope_theta=theta)
    seq = torch.arange(nseq, **i32)
    cu = torch.arange(nseq + 1, **i32) * S
    cache.append(seq, q_start, cu, k.flatten(0, 1), v.flatten(0, 1))

    # generation: three fused steps
    pos = np.full(nseq, S)
    for _ in range(3):
        kk, vv = kv_at(pos)
        o, l = cache.decode_append(bits_to_bf16_tensor(q_at(pos)), bits_to_bf16_tensor(kk),
                                   bits_to_bf16_tensor(vv), torch.tensor(pos, **i32))
        torch.cuda.synchronize()
        check(o, l, pos, f"decode at {pos[0]}")
        pos = pos + 1

    # one more step through the executor, inputs and results in pinned host memory
    g = ps.DecodeGraph(cache, hq)
    host_in = torch.zeros(g.inp.numel(), dtype=torch.uint8).pin_memory()
    host_res = torch.zeros(g.res.numel(), dtype=torch.uint8).pin_memory()
    kk, vv = kv_at(pos)
    for name, bits in (("q", q_at(pos)), ("k", kk), ("v", vv)):
        o_, n_ = g.in_layout[name]
        host_in[o_:o_ + n_] = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8).reshape(-1))
    o_, n_ = g.in_layout["pos"]
    host_in[o_:o_ + n_] = torch.from_numpy(pos.astype(np.int32).view(np.uint8))
    g.step(host_in, host_res)
    o_, n_ = g.res_layout["out"]
    o = host_res[o_:o_ + n_].view(torch.bfloat16).view(nseq, hq, D)
    o_, n_ = g.res_layout["lse"]
    l = host_res[o_:o_ + n_].view(torch.float32).view(nseq, hq)
    check(o, l, pos, "executor step")
    assert cache.check_status() == 0
    g.close()
