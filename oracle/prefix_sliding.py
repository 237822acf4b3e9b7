"""Plain float64 CPU oracle for Prefix-Sliding attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library never does.

It computes the definition of the method directly, from the full,
never-evicted K/V history, one query row at a time, with no blocking, fusion
or reordering.  Sources (page title, then the section or paragraph):

[NJH]  njhaofan.com article on PrefixSliding, section
       "PrefixSliding如何丢掉中间Token？" (fixed prefix + last-W window, the
       4196-token cap, Continue PE, tile skipping in the Hopper kernel).
[EXP]  "Prefix Sliding：面向高效 test-time scaling 的前缀滑动方法"
       (papers.ananclaw.com), sections "核心方法" and "伪代码" (PREFIX and
       WINDOW blocks; cache size is the constant prefix_len + W).
[AGI]  "Prefix Sliding for efficient test-time scaling" (agihunt.info), the
       paragraphs on the 100-token prefix + 4,096 window cap, on Continue PE,
       and on the two-level tile filter of the FlashAttention kernel.

Readings taken where the pages are silent (each is restated where it is used):
  * the window includes the current token: query p sees key j iff
    j <= p and (j < P or j > p - W), so at most P + W keys ([NJH], [AGI] cap
    of 100 + 4096 = 4196);
  * RoPE is the half-split ("NeoX") rotation with inv_freq_i = theta^(-2i/D),
    applied at the absolute, ever-increasing position (Continue PE, [AGI]);
  * rotated Q and K are rounded to bfloat16 (the cache stores bfloat16);
    values V are used as given;
  * softmax scale 1/sqrt(D), LSE is the natural log of sum(exp(score)),
    query head h reads KV head h // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np

SKIP, PARTIAL, FULL = 0, 1, 2


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits and float32's exponent range; below
    2**-126 the spacing is fixed at 2**-133 (subnormals).  One rounding from
    the exact float64 value.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # subnormal range keeps a fixed quantum
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(x / quantum) * quantum       # rint: round half to even
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, x), r)
    return np.where(x == 0.0, x, r)


# --------------------------------------------------------------------------
# RoPE with Continue PE ([AGI] paragraph on position encodings)
# --------------------------------------------------------------------------
def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate the last axis (length D, even) of ``x`` at absolute position(s) ``pos``.

    Half-split pairing: element i rotates with element i + D/2 by the angle
    pos * theta**(-2i/D).  ``pos`` broadcasts against the leading axes of ``x``
    (a scalar, or one position per leading row).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    p = np.asarray(pos, dtype=np.float64)
    p = p.reshape(p.shape + (1,) * (x.ndim - p.ndim))   # align to x's leading axes
    ang = p * inv_freq                                   # broadcasts over the last axis
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------
# the mask ([NJH] section "PrefixSliding如何丢掉中间Token？", [EXP] "核心方法")
# --------------------------------------------------------------------------
def allowed(p, j, P: int, W: int):
    """True where query position p may attend key position j."""
    p = np.asarray(p)
    j = np.asarray(j)
    return (j <= p) & ((j < P) | (j > p - W))


def visible_positions(p: int, P: int, W: int) -> np.ndarray:
    """All key positions query p sees, found by scanning the whole history [0, p]."""
    j = np.arange(p + 1, dtype=np.int64)
    return j[allowed(p, j, P, W)]


# --------------------------------------------------------------------------
# attention over an explicit key set
# --------------------------------------------------------------------------
def masked_attention(q_hat, k_hat, v, scale: float):
    """Softmax attention of each query head over every given key (float64).

    q_hat [Hq, D]; k_hat, v [n, Hkv, D].  Returns O [Hq, D] and the natural-log
    LSE [Hq] of the scaled scores.
    """
    q_hat = np.asarray(q_hat, dtype=np.float64)
    hq = q_hat.shape[0]
    hkv = k_hat.shape[1]
    group = hq // hkv
    out = np.zeros((hq, v.shape[2]))
    lse = np.zeros(hq)
    for h in range(hq):
        kh = h // group
        s = (k_hat[:, kh, :] @ q_hat[h]) * scale
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        lse[h] = m + math.log(l)
        out[h] = (e / l) @ v[:, kh, :]
    return out, lse


def attend(q_raw, p: int, P: int, W: int, history, theta: float, scale: float | None = None):
    """Prefix-Sliding attention output of one query at absolute position p.

    ``q_raw`` [Hq, D] float64 (raw bfloat16 values, before RoPE).
    ``history(positions)`` returns raw k, v [n, Hkv, D] float64 at those
    absolute positions; the oracle asks only for the positions the mask admits,
    after scanning every j in [0, p].
    """
    q_raw = np.asarray(q_raw, dtype=np.float64)
    d = q_raw.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    js = visible_positions(p, P, W)
    k_raw, v = history(js)
    q_hat = round_bf16(rope(q_raw, p, theta))
    k_hat = round_bf16(rope(k_raw, js, theta))
    return masked_attention(q_hat, k_hat, v, scale)


def reset_positions(p: int, P: int, W: int) -> tuple[np.ndarray, np.ndarray, int]:
    """Reset PE renumbering for query p ([AGI] paragraph on position encodings:
    Reset PE reassigns the cached entries' positions; the pages do not give the
    rule).  Reading taken: the cache is renumbered in order, the P prefix keys
    keep 0..P-1 and the window keys, oldest first, take P, P+1, ...; the query
    is the newest window entry.  Returns (key positions js, their reset
    positions, the query's reset position)."""
    js = visible_positions(p, P, W)
    reset = np.where(js < P, js, 0)
    win = js >= P
    reset[win] = P + np.arange(int(win.sum()))
    return js, reset, int(reset[-1])


def attend_reset_pe(q_raw, p: int, P: int, W: int, history, theta: float,
                    scale: float | None = None):
    """Prefix-Sliding attention of query p under Reset PE.

    The scores depend only on the rotation between query and key, so a key
    kept rotated at its absolute position j (the cache is never rewritten) and
    a query rotated at r_q - (r_j - j), with r the reset positions, give the
    reset-position score exactly.  Window keys are contiguous, so r_q - r_j =
    p - j for them: their query rotation is the absolute one, p.  Prefix keys
    keep r_j = j: their query rotation is r_q.  Rounding contract as in
    ``attend``: the stored key and each rotated query are bf16.
    """
    q_raw = np.asarray(q_raw, dtype=np.float64)
    d = q_raw.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    js, reset, rq = reset_positions(p, P, W)
    k_raw, v = history(js)
    k_hat = round_bf16(rope(k_raw, js, theta))
    q_win = round_bf16(rope(q_raw, p, theta))
    q_pre = round_bf16(rope(q_raw, rq, theta))
    pre = js < P
    hq = q_raw.shape[0]
    group = hq // k_hat.shape[1]
    out = np.zeros((hq, d))
    lse = np.zeros(hq)
    for h in range(hq):
        kh = h // group
        s = np.where(pre, k_hat[:, kh, :] @ q_pre[h], k_hat[:, kh, :] @ q_win[h]) * scale
        m = s.max()
        e = np.exp(s - m)
        lse[h] = m + math.log(e.sum())
        out[h] = (e / e.sum()) @ v[:, kh, :]
    return out, lse


# --------------------------------------------------------------------------
# backward of the training forward ([AGI] paragraph on truncated backprop:
# the trainer back-propagates through the last 4W tokens under the mask)
# --------------------------------------------------------------------------
def attend_backward(q_raw, k_raw, v, d_out, P: int, W: int, theta: float,
                    scale: float | None = None, positions=None):
    """Gradients of Prefix-Sliding attention over one sequence (float64).

    q_raw [S, Hq, D], k_raw / v [S, Hkv, D] (raw values), d_out [S, Hq, D]
    (gradient of the loss w.r.t. O); positions default to 0..S-1.  Forward as
    in ``attend``: q_hat = bf16(rope(q)), k_hat = bf16(rope(k)), softmax of
    scale * q_hat . k_hat over the admitted keys.  Backward, per query row i
    and admitted key j:
        P_ij = exp(s_ij - LSE_i),   dV_j += P_ij dO_i,
        dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij = dO_i . O_i,
        dS_ij = P_ij (dP_ij - D_i),
        dQhat_i = scale sum_j dS_ij k_hat_j,   dKhat_j += scale dS_ij q_hat_i,
    then back through the rotation (its transpose is the rotation by the
    negative angle); the bf16 rounding passes gradients straight through.
    Query head h reads KV head h // (Hq / Hkv), so dK and dV sum over the
    group.  Returns (dq_raw, dk_raw, dv, O, LSE [S, Hq]).
    """
    q_raw = np.asarray(q_raw, dtype=np.float64)
    k_raw = np.asarray(k_raw, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_out = np.asarray(d_out, dtype=np.float64)
    S, hq, d = q_raw.shape
    hkv = k_raw.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.arange(S) if positions is None else np.asarray(positions)
    q_hat = round_bf16(rope(q_raw, pos, theta))
    k_hat = round_bf16(rope(k_raw, pos, theta))
    dq_hat = np.zeros_like(q_hat)
    dk_hat = np.zeros_like(k_hat)
    dv = np.zeros_like(v)
    out = np.zeros_like(q_raw)
    lse = np.zeros((S, hq))
    for i in range(S):
        js = np.nonzero(allowed(pos[i], pos, P, W))[0]
        for h in range(hq):
            kh = h // group
            s = (k_hat[js, kh, :] @ q_hat[i, h]) * scale
            m = s.max()
            e = np.exp(s - m)
            lse[i, h] = m + math.log(e.sum())
            pr = np.exp(s - lse[i, h])
            out[i, h] = pr @ v[js, kh, :]
            dv[js, kh, :] += np.outer(pr, d_out[i, h])
            dp = v[js, kh, :] @ d_out[i, h]
            ds = pr * (dp - pr @ dp)
            dq_hat[i, h] = scale * (ds @ k_hat[js, kh, :])
            dk_hat[js, kh, :] += scale * np.outer(ds, q_hat[i, h])
    dq_raw = rope(dq_hat, -pos, theta)
    dk_raw = rope(dk_hat, -pos, theta)
    return dq_raw, dk_raw, dv, out, lse


def attend_backward_at(q_raw, k_raw, v, d_out, P: int, W: int, theta: float, q_rows, k_rows,
                       scale: float | None = None, positions=None, rows_per_pass: int = 64):
    """Selected rows of the gradients ``attend_backward`` returns, for sequences
    too long to form all of them: dq at the query rows ``q_rows`` and dk, dv at
    the key rows ``k_rows``.

    Same forward, rounding contract and backward formulas as
    ``attend_backward``.  A query row's dq needs only that row's softmax; a
    key's dk and dv need every query row that admits the key.  So the function
    visits the rows of ``q_rows`` and every row that admits one of ``k_rows``.
    For each visited row i and query head h it forms the scores against every
    key of the sequence, sets the ones the mask refuses to -inf (weight 0), and
    takes P, dP, D_i and dS as ``attend_backward`` does.  Rows are independent;
    ``rows_per_pass`` of them go through each matrix product together.
    Returns dq [len(q_rows), Hq, D], dk and dv [len(k_rows), Hkv, D].
    """
    q_raw = np.asarray(q_raw, dtype=np.float64)
    k_raw = np.asarray(k_raw, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_out = np.asarray(d_out, dtype=np.float64)
    S, hq, d = q_raw.shape
    hkv = k_raw.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.arange(S) if positions is None else np.asarray(positions)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    q_hat = round_bf16(rope(q_raw, pos, theta))
    k_hat = round_bf16(rope(k_raw, pos, theta))
    dq_hat = np.zeros((len(q_rows), hq, d))
    dk_hat = np.zeros((len(k_rows), hkv, d))
    dv = np.zeros((len(k_rows), hkv, d))
    need = set(q_rows.tolist())
    for j in k_rows:
        need.update(np.nonzero(allowed(pos, pos[j], P, W))[0].tolist())
    need = np.array(sorted(need), dtype=np.int64)
    for a in range(0, len(need), rows_per_pass):
        rows = need[a:a + rows_per_pass]
        keep = allowed(pos[rows][:, None], pos[None, :], P, W)         # [R, S]
        for kv in range(hkv):
            for h in range(kv * group, (kv + 1) * group):
                s = (q_hat[rows, h, :] @ k_hat[:, kv, :].T) * scale     # [R, S]
                s = np.where(keep, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                lse = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))
                pr = np.exp(s - lse)
                dp = d_out[rows, h, :] @ v[:, kv, :].T
                ds = pr * (dp - (pr * dp).sum(axis=1, keepdims=True))
                for r, i in enumerate(rows):
                    for n in np.nonzero(q_rows == i)[0]:
                        dq_hat[n, h] = scale * (ds[r] @ k_hat[:, kv, :])
                for n, j in enumerate(k_rows):
                    dk_hat[n, kv] += scale * (ds[:, j] @ q_hat[rows, h, :])
                    dv[n, kv] += pr[:, j] @ d_out[rows, h, :]
    dq = rope(dq_hat, -pos[q_rows], theta)
    dk = rope(dk_hat, -pos[k_rows], theta)
    return dq, dk, dv


# --------------------------------------------------------------------------
# the bounded cache ([EXP] "伪代码" invariant: size prefix_len + W)
# --------------------------------------------------------------------------
def ring_slot(pos: int, P: int, W: int) -> int:
    """Slot of absolute position pos in a cache of P fixed + W rotating slots."""
    return pos if pos < P else P + (pos - P) % W


class RingSim:
    """Position-level simulation of the P + W slot cache.

    Each append stores the position in its slot.  ``check(p)`` asserts that
    the positions held after appending 0..p are exactly the ones query p may
    see by the mask definition.
    """

    def __init__(self, P: int, W: int):
        self.P, self.W = P, W
        self.slots = np.full(P + W, -1, dtype=np.int64)

    def append(self, pos: int) -> int:
        s = ring_slot(pos, self.P, self.W)
        self.slots[s] = pos
        return s

    def live(self) -> np.ndarray:
        return np.sort(self.slots[self.slots >= 0])

    def check(self, p: int) -> None:
        want = visible_positions(p, self.P, self.W)
        got = self.live()
        if not np.array_equal(got, want):
            raise AssertionError(f"ring holds {got} but query {p} sees {want}")


# --------------------------------------------------------------------------
# tile classes ([NJH] / [AGI]: skip tiles wholly outside prefix and window,
# mask elementwise inside tiles that straddle the boundary)
# --------------------------------------------------------------------------
def tile_classes(q_pos, k_pos, P: int, W: int, BM: int, BN: int) -> np.ndarray:
    """Brute-force class of each (query tile, key tile): SKIP, PARTIAL or FULL.

    ``q_pos`` / ``k_pos`` are the absolute positions of the query rows and of
    the key rows in array order; tile (a, b) holds rows [a*BM, (a+1)*BM) and
    keys [b*BN, (b+1)*BN), clipped to the arrays.  SKIP: no admitted pair;
    FULL: every pair admitted; PARTIAL: otherwise.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    nq = -(-len(q_pos) // BM)
    nk = -(-len(k_pos) // BN)
    out = np.zeros((nq, nk), dtype=np.uint8)
    for a in range(nq):
        qs = q_pos[a * BM:(a + 1) * BM]
        m = allowed(qs[:, None], k_pos[None, :], P, W)
        for b in range(nk):
            blk = m[:, b * BN:(b + 1) * BN]
            out[a, b] = FULL if blk.all() else (PARTIAL if blk.any() else SKIP)
    return out
