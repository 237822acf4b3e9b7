"""ps_prefill_backward (dq, dk, dv) against the float64 oracle's gradients (GPU).

Tolerance: the kernels feed the probabilities and dS to the tensor cores as
bf16 (relative rounding 2^-9 per element) and start from the forward's bf16
O and fp32 LSE, so each gradient tensor is compared per head against the
oracle as max|g - g_ref| <= 2e-2 * max|g_ref|, with the mean error held to a
tenth of that.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attend_backward

from _util import bits_to_bf16_tensor

pytestmark = pytest.mark.gpu

STREAM_DO = 5  # synthetic dO


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def _close(g, ref, what):
    """g, ref: [S, H, D] float64; checked per head."""
    for h in range(ref.shape[1]):
        scale = float(np.abs(ref[:, h]).max())
        err = np.abs(g[:, h] - ref[:, h])
        assert err.max() <= 2e-2 * scale, f"{what} head {h}: max err {err.max():.3e} vs max {scale:.3e}"
        assert err.mean() <= 2e-3 * scale, f"{what} head {h}: mean err {err.mean():.3e} vs max {scale:.3e}"


@pytest.mark.parametrize("B,S,hq,hkv,P,W,D", [
    (1, 300, 4, 2, [37], 100, 128),        # ragged tail, prefix and band
    (1, 300, 4, 2, [37], 100, 64),    # the same at head_dim 64
    (2, 257, 2, 2, [5, 0], 1000, 128),     # one query head per KV head; W >= S: causal
    (1, 384, 8, 2, [0], 128, 128),         # G = 4; plain sliding window
    (1, 200, 4, 2, [300], 16, 128),        # P >= S: causal through the prefix
    (2, 1024, 16, 8, [64, 64], 256, 128),  # training-shaped, reduced: 4W tokens, loss on all
    (1, 300, 8, 1, [37], 100, 128),        # G = 8: one dK/dV CTA sums eight query heads
    (1, 300, 6, 2, [37], 100, 128),        # G = 3 (odd group)
])
def test_backward_matches_oracle(ps, B, S, hq, hkv, P, W, D):
    seed, theta = 41, 10000.0
    pos = np.arange(S)
    q = np.stack([synth.query_bits(seed, b, pos, hq, D) for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(pos) for b in range(B)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    do = np.stack([synth.normal_bf16(seed, STREAM_DO, b, pos, hq, D) for b in range(B)])
    i32 = dict(dtype=torch.int32, device="cuda")
    tq, tk, tv, tdo = (bits_to_bf16_tensor(x) for x in (q, k, v, do))
    qs = torch.zeros(B, **i32)
    pl = torch.tensor(P, **i32)
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
    dq, dk, dv = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(B):
        rq, rk, rv, _, _ = attend_backward(synth.bits_to_f64(q[b]), synth.bits_to_f64(k[b]),
                                           synth.bits_to_f64(v[b]), synth.bits_to_f64(do[b]),
                                           P[b], W, theta)
        _close(dq[b].double().cpu().numpy(), rq, f"dq b={b}")
        _close(dk[b].double().cpu().numpy(), rk, f"dk b={b}")
        _close(dv[b].double().cpu().numpy(), rv, f"dv b={b}")


@pytest.mark.parametrize("B,S,hq,hkv,P,W,c0", [
    (2, 300, 4, 2, [100, 100], 64, [50, 1000]),  # chunk starts inside / after the prefix
    (1, 256, 2, 1, [40], 128, [7]),              # unaligned start: RoPE at odd positions
])
def test_backward_chunk_offset(ps, B, S, hq, hkv, P, W, c0):
    """A chunk at positions q_start .. q_start + S - 1 (no cached history): the mask
    and the rotations use absolute positions."""
    seed, D, theta = 43, 128, 10000.0
    pos = [c + np.arange(S) for c in c0]
    q = np.stack([synth.query_bits(seed, b, pos[b], hq, D) for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(pos[b]) for b in range(B)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    do = np.stack([synth.normal_bf16(seed, STREAM_DO, b, pos[b], hq, D) for b in range(B)])
    i32 = dict(dtype=torch.int32, device="cuda")
    tq, tk, tv, tdo = (bits_to_bf16_tensor(x) for x in (q, k, v, do))
    qs = torch.tensor(c0, **i32)
    pl = torch.tensor(P, **i32)
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
    dq, dk, dv = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(B):
        rq, rk, rv, _, _ = attend_backward(synth.bits_to_f64(q[b]), synth.bits_to_f64(k[b]),
                                           synth.bits_to_f64(v[b]), synth.bits_to_f64(do[b]),
                                           P[b], W, theta, positions=pos[b])
        _close(dq[b].double().cpu().numpy(), rq, f"dq b={b}")
        _close(dk[b].double().cpu().numpy(), rk, f"dk b={b}")
        _close(dv[b].double().cpu().numpy(), rv, f"dv b={b}")


def test_training_backward_full_size_sampled():
    """The 8 x 8,192 training backward (P = 256, W = 2,048, 16/8 heads) in the launch
    configuration the benchmark times.  Batch row 0: dq at the mask's edges and
    dk, dv of prefix keys, band keys and the last key (these need every query row
    that sees them).  Batch row 7: dq rows only.  The oracle's selected-row
    gradients use the same formulas as its whole-sequence ones."""
    import prefix_sliding_window_02_b300 as ps
    from oracle import attend_backward_at
    seed, B, S, hq, hkv, D, P, W, theta = 42, 8, 8192, 16, 8, 128, 256, 2048, 10000.0
    pos = np.arange(S)
    q = np.stack([synth.query_bits(seed, b, pos, hq, D) for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(pos) for b in range(B)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    do = np.stack([synth.normal_bf16(seed, STREAM_DO, b, pos, hq, D) for b in range(B)])
    i32 = dict(dtype=torch.int32, device="cuda")
    tq, tk, tv, tdo = (bits_to_bf16_tensor(x) for x in (q, k, v, do))
    qs = torch.zeros(B, **i32)
    pl = torch.full((B,), P, **i32)
    status = torch.zeros(1, **i32)
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, status=status)
    dq, dk, dv = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert all(torch.isfinite(g).all() for g in (dq, dk, dv))
    rng = np.random.default_rng(7)
    q_rows = sorted(set([0, 1, 127, 128, 255, 256, 2047, 2048, 2303, 2304, 4095, 8191]
                        + rng.integers(0, S, 6).tolist()))
    samples = {0: (q_rows, [0, 131, 255, 256, 2047, 2048, 5000, 8190, 8191]), 7: (q_rows, [])}
    for b, (qr, kr) in samples.items():
        rq, rk, rv = attend_backward_at(synth.bits_to_f64(q[b]), synth.bits_to_f64(k[b]),
                                        synth.bits_to_f64(v[b]), synth.bits_to_f64(do[b]), P, W,
                                        theta, qr, kr)
        _close(dq[b, qr].double().cpu().numpy(), rq, f"dq b={b}")
        if kr:
            _close(dk[b, kr].double().cpu().numpy(), rk, f"dk b={b}")
            _close(dv[b, kr].double().cpu().numpy(), rv, f"dv b={b}")


@pytest.mark.parametrize("D", [128, 64])
def test_backward_reuses_forward_rotations_bit_exactly(D):
    """Given the forward's workspace, the backward reads the rotated Q and K the
    forward left there instead of rotating again: the gradients are the same bits."""
    import prefix_sliding_window_02_b300 as ps
    seed, B, S, hq, hkv, P, W, theta = 44, 2, 700, 4, 2, [37, 300], 128, 10000.0
    pos = np.arange(S)
    q = np.stack([synth.query_bits(seed, b, pos, hq, D) for b in range(B)])
    kv = [synth.History(seed, b, hkv, D).rows_bits(pos) for b in range(B)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    do = np.stack([synth.normal_bf16(seed, STREAM_DO, b, pos, hq, D) for b in range(B)])
    i32 = dict(dtype=torch.int32, device="cuda")
    tq, tk, tv, tdo = (bits_to_bf16_tensor(x) for x in (q, k, v, do))
    qs = torch.tensor([0, 50], **i32)
    pl = torch.tensor(P, **i32)
    status = torch.zeros(1, **i32)
    ws = torch.empty(ps.prefill_workspace_size(B, S, hq, hkv, D), dtype=torch.uint8, device="cuda")
    out, lse = ps.prefill(tq, tk, tv, qs, pl, W, rope_theta=theta, workspace=ws, status=status)
    a = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta, status=status)
    b = ps.prefill_backward(tq, tk, tv, out, lse, tdo, qs, pl, W, rope_theta=theta, status=status,
                            fwd_workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, y in zip(a, b):
        assert torch.equal(x, y)
