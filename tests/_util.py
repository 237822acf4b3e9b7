"""Shared helpers for the GPU parity tests (input plumbing and tolerances)."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Tolerances for bf16 inputs with fp32 accumulation (per (case, head) tensor):
O_ABS = 1e-2      # max |O_gpu - O_ref|
O_REL = 2e-2      # max |O_gpu - O_ref| / max |O_ref|
LSE_ABS = 1e-3    # max |LSE_gpu - LSE_ref|


def bits_to_bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def live_runs(p: int, P: int, W: int):
    """Runs (first_position, length) whose tokens a cache holds after 0..p."""
    if p + 1 <= P + W:
        return [(0, p + 1)]
    runs = [(0, P)] if P > 0 else []
    runs.append((p - W + 1, W))
    return runs


def append_runs(cache, runs_per_seq, kv_source, device="cuda"):
    """Append, for every sequence, its list of (pos0, n) runs.

    kv_source(s, positions) -> (k_bits or tensor, v_bits or tensor) [n, Hkv, D].
    Runs with the same index in each sequence's list go in one call, so one
    call never holds two runs of the same sequence.
    """
    depth = max(len(r) for r in runs_per_seq.values())
    for i in range(depth):
        seqs, pos0, cu, ks, vs = [], [], [0], [], []
        for s, runs in runs_per_seq.items():
            if i >= len(runs) or runs[i][1] == 0:
                continue
            a, n = runs[i]
            k, v = kv_source(s, np.arange(a, a + n))
            if isinstance(k, np.ndarray):
                k, v = bits_to_bf16_tensor(k, device), bits_to_bf16_tensor(v, device)
            seqs.append(s)
            pos0.append(a)
            cu.append(cu[-1] + n)
            ks.append(k)
            vs.append(v)
        if not seqs:
            continue
        i32 = dict(dtype=torch.int32, device=device)
        cache.append(torch.tensor(seqs, **i32), torch.tensor(pos0, **i32), torch.tensor(cu, **i32),
                     torch.cat(ks).contiguous(), torch.cat(vs).contiguous())


def synth_source(seed, hkv, d):
    def src(s, pos):
        return synth.History(seed, s, hkv, d).rows_bits(pos)
    return src


def random_source(seed, hkv, d, device="cuda"):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def src(s, pos):
        n = len(pos)
        k = torch.randn(n, hkv, d, generator=gen, device=device).to(torch.bfloat16)
        v = torch.randn(n, hkv, d, generator=gen, device=device).to(torch.bfloat16)
        return k, v
    return src


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_*: [H, D]; lse_*: [H].  Checks each head against the stated tolerances."""
    for h in range(o_ref.shape[0]):
        d = float(np.abs(o_gpu[h] - o_ref[h]).max())
        ref = float(np.abs(o_ref[h]).max())
        dl = float(abs(lse_gpu[h] - lse_ref[h]))
        assert d <= O_ABS, f"{what} head {h}: max|dO| = {d:.3e}"
        assert d <= O_REL * ref, f"{what} head {h}: max|dO|/max|O| = {d / ref:.3e}"
        assert dl <= LSE_ABS, f"{what} head {h}: |dLSE| = {dl:.3e}"
