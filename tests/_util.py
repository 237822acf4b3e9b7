"""Shared helpers for the GPU parity tests (input plumbing and tolerances)."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Tolerances for bf16 inputs with fp32 accumulation, read as an absolute plus a
# relative term per element (the numpy/torch allclose convention):
#     |O_gpu - O_ref| <= O_ABS + O_REL * |O_ref|   and   |LSE_gpu - LSE_ref| <= LSE_ABS.
# O is returned in bf16, whose rounding alone is half an ulp of the value
# (0.0156 for |O| in [4, 8)), so a purely absolute 1e-2 bound cannot hold for
# large outputs of any bf16-output kernel; the relative term covers that.
O_ABS = 1e-2
O_REL = 2e-2
LSE_ABS = 1e-3


def lse_tol(qscale_log2: int = 0) -> float:
    """LSE bound for queries scaled by 2**qscale_log2 (stress cases only).

    Both sides round the rotated query to bf16; the kernel rotates in fp32 and
    the oracle in fp64, so an element lying almost exactly between two bf16
    values can round to different neighbours (about one element in 10^4).  One
    such flip moves a score by one bf16 ulp of q_i times |k_i| / sqrt(D), and
    the LSE of a row dominated by that key by the same amount; scaling q by 2^s
    scales the ulp, hence the bound, by 2^s.  Unscaled inputs keep 1e-3.
    """
    return LSE_ABS * 2.0 ** qscale_log2


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


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", lse_abs=LSE_ABS):
    """o_*: [H, D]; lse_*: [H].  Checks each head against the stated tolerances."""
    for h in range(o_ref.shape[0]):
        err = np.abs(o_gpu[h] - o_ref[h])
        bound = O_ABS + O_REL * np.abs(o_ref[h])
        i = int(np.argmax(err - bound))
        dl = float(abs(lse_gpu[h] - lse_ref[h]))
        assert err[i] <= bound[i], (f"{what} head {h}: |dO| = {err[i]:.3e} at element {i} "
                                    f"(|O_ref| = {abs(o_ref[h][i]):.3e}, bound {bound[i]:.3e})")
        assert dl <= lse_abs, f"{what} head {h}: |dLSE| = {dl:.3e}"
