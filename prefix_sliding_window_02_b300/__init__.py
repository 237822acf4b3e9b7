"""Prefix-Sliding attention on B300: Python binding of libps.so.

Argument marshalling only: every step runs in the library's CUDA kernels.
torch supplies device memory and streams.  Names follow include/ps.h.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from ._lib import (CacheDesc, PsError, StepLayout, check, lib,  # noqa: F401
                   PS_DEV_BAD_POS, PS_DEV_BAD_PREFIX, PS_DEV_BAD_RUN, PS_DEV_BAD_SEQ,
                   PS_DEV_BAD_SLOT, PS_DEV_TIMEOUT, PS_PE_CONTINUE, PS_PE_RESET)

__all__ = ["RingCache", "DecodeGraph", "decode_step_layout", "ring_slots", "decode_workspace_size",
           "prefill_workspace_size", "prefill", "prefill_backward", "prefill_tile_grid",
           "prefill_tile_classes", "PsError", "lib"]

BF16 = torch.bfloat16


def _vp(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}, got "
                         f"{t.dtype} on {t.device} (contiguous={t.is_contiguous()})")


def _shape(t: torch.Tensor, shape, name: str):
    """The library trusts the sizes it is given: check every tensor against the
    shape the call implies before any pointer reaches it."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _dims(t: torch.Tensor, n: int, name: str, what: str):
    if t.dim() != n:
        raise ValueError(f"{name}: expected {what}, got shape {tuple(t.shape)}")


class RingCache:
    """Bounded per-sequence K/V cache of ``prefix_max + window`` slots.

    Contiguous (default): pools of shape [nseq * capacity, n_kv_heads, head_dim];
    sequence s owns rows [s * capacity, (s + 1) * capacity).
    ``pe_mode``: PS_PE_CONTINUE (0, the default) or PS_PE_RESET (1), the
    position encoding ps_decode applies (see include/ps.h).
    Paged (``block_size`` given, a multiple of 16): the pools hold
    ``nseq * blocks_per_seq`` blocks of ``block_size`` rows, and
    ``block_table[s, i]`` names the block of the sequence's logical slots
    [i * block_size, (i + 1) * block_size); ``block_order`` (a permutation of the
    block ids, default identity) sets that assignment.
    ``slot_base`` (contiguous only): the first pool row of each sequence instead of
    ``s * capacity``; the pools then hold ``max(slot_base) + capacity`` rows.
    Sequences touch only the rows of the slots they fill, so reservations may
    overlap where a sequence never fills its whole capacity (e.g. a full-history
    cache whose sequences stop at different positions).
    """

    def __init__(self, nseq: int, n_kv_heads: int, head_dim: int, window: int,
                 prefix_len: Sequence[int] | torch.Tensor, rope_theta: float = 10000.0,
                 prefix_max: Optional[int] = None, capacity: Optional[int] = None,
                 device="cuda", zero: bool = True, block_size: Optional[int] = None,
                 block_order: Optional[Sequence[int]] = None, pe_mode: int = 0,
                 slot_base: Optional[Sequence[int]] = None):
        pl = torch.as_tensor(prefix_len, dtype=torch.int32).reshape(-1)
        if pl.numel() != nseq:
            raise ValueError("prefix_len must have nseq entries")
        self.prefix_max = int(pl.max()) if prefix_max is None else int(prefix_max)
        self.capacity = self.prefix_max + window if capacity is None else int(capacity)
        self.nseq, self.n_kv_heads, self.head_dim, self.window = nseq, n_kv_heads, head_dim, window
        self.rope_theta = float(rope_theta)
        self.block_size = block_size
        if slot_base is not None and block_size is not None:
            raise ValueError("slot_base applies to contiguous caches only")
        if slot_base is not None:
            base = torch.as_tensor(slot_base, dtype=torch.int64).reshape(-1)
            if base.numel() != nseq or int(base.min()) < 0:
                raise ValueError("slot_base must have nseq non-negative entries")
        else:
            base = torch.arange(nseq, dtype=torch.int64) * self.capacity
        self._base = base
        if block_size is None:
            rows = int(base.max()) + self.capacity
            self.block_table = None
            self.blocks_per_seq = 0
        else:
            self.blocks_per_seq = -(-self.capacity // block_size)
            nblocks = nseq * self.blocks_per_seq
            rows = nblocks * block_size
            order = torch.arange(nblocks, dtype=torch.int32) if block_order is None else \
                torch.as_tensor(block_order, dtype=torch.int32)
            if sorted(order.tolist()) != list(range(nblocks)):
                raise ValueError("block_order must be a permutation of the block ids")
            self.block_table = order.reshape(nseq, self.blocks_per_seq).contiguous().to(device)
        alloc = torch.zeros if zero else torch.empty
        self.k_pool = alloc(rows, n_kv_heads, head_dim, dtype=BF16, device=device)
        self.v_pool = alloc(rows, n_kv_heads, head_dim, dtype=BF16, device=device)
        self.slot_base = base.to(device)
        self.prefix_len = pl.to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self._ws = None
        self.desc = CacheDesc(
            k_pool=self.k_pool.data_ptr(), v_pool=self.v_pool.data_ptr(),
            slot_base=self.slot_base.data_ptr(), prefix_len=self.prefix_len.data_ptr(),
            status=self.status.data_ptr(), total_slots=rows, nseq=nseq, n_kv_heads=n_kv_heads,
            head_dim=head_dim, window=window, capacity=self.capacity, prefix_max=self.prefix_max,
            rope_theta=self.rope_theta,
            block_table=None if self.block_table is None else self.block_table.data_ptr(),
            block_size=block_size or 0, blocks_per_seq=self.blocks_per_seq, pe_mode=pe_mode)
        self.pe_mode = pe_mode

    def rows_of(self, seq: int) -> torch.Tensor:
        """Pool rows of the sequence's logical slots 0..capacity-1, in slot order."""
        slots = torch.arange(self.capacity, dtype=torch.int64)
        if self.block_table is None:
            return int(self._base[seq]) + slots
        bt = self.block_table[seq].cpu().to(torch.int64)
        return bt[slots // self.block_size] * self.block_size + slots % self.block_size

    # ------------------------------------------------------------ append ----
    def append(self, seq_idx: torch.Tensor, pos0: torch.Tensor, cu_tokens: torch.Tensor,
               k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        """ps_kv_append: runs r = tokens [cu[r], cu[r+1]) of sequence seq_idx[r]
        at positions pos0[r], pos0[r] + 1, ...  k, v: [n_tokens, Hkv, D] bf16, raw."""
        _dims(k, 3, "k", "[n_tokens, Hkv, D]")
        _dims(seq_idx, 1, "seq_idx", "[n_runs]")
        n_tok, n_runs = k.shape[0], seq_idx.shape[0]
        _shape(k, (n_tok, self.n_kv_heads, self.head_dim), "k")
        _shape(v, (n_tok, self.n_kv_heads, self.head_dim), "v")
        _shape(pos0, (n_runs,), "pos0")
        _shape(cu_tokens, (n_runs + 1,), "cu_tokens")
        for t, n in ((seq_idx, "seq_idx"), (pos0, "pos0"), (cu_tokens, "cu_tokens")):
            _need(t, torch.int32, n)
        _need(k, BF16, "k")
        _need(v, BF16, "v")
        check(lib.ps_kv_append(ctypes.byref(self.desc), _vp(seq_idx), _vp(pos0), _vp(cu_tokens),
                               seq_idx.numel(), _vp(k), _vp(v), k.shape[0], _stream(stream)),
              "ps_kv_append")

    def append_tokens(self, pos: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None,
                      _cu: dict = {}) -> None:
        """One token per sequence (the decode step): k, v [nseq, Hkv, D], pos [nseq]."""
        _shape(pos, (self.nseq,), "pos")
        _shape(k, (self.nseq, self.n_kv_heads, self.head_dim), "k")
        key = (self.nseq, k.device)
        if key not in _cu:
            _cu[key] = (torch.arange(self.nseq, dtype=torch.int32, device=k.device),
                        torch.arange(self.nseq + 1, dtype=torch.int32, device=k.device))
        seq, cu = _cu[key]
        self.append(seq, pos, cu, k, v, stream)

    # ------------------------------------------------------------ decode ----
    def _check_q(self, q: torch.Tensor, pos: torch.Tensor) -> int:
        _dims(q, 3, "q", "[nseq, Hq, D]")
        _shape(q, (self.nseq, q.shape[1], self.head_dim), "q")
        _shape(pos, (self.nseq,), "pos")
        return q.shape[1]

    def workspace(self, n_q_heads: int) -> torch.Tensor:
        need = decode_workspace_size(self.nseq, n_q_heads, self.n_kv_heads, self.head_dim)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.k_pool.device)
        return self._ws

    def decode(self, q: torch.Tensor, pos: torch.Tensor, scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None):
        """ps_decode: q [nseq, Hq, D] bf16 raw; pos [nseq] int32.  Returns (out, lse)."""
        hq = self._check_q(q, pos)
        if out is not None:
            _shape(out, q.shape, "out")
        if lse is not None:
            _shape(lse, (self.nseq, hq), "lse")
        _need(q, BF16, "q")
        _need(pos, torch.int32, "pos")
        if scale is None:
            scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(q.shape[0], hq, dtype=torch.float32, device=q.device)
        ws = self.workspace(hq) if workspace is None else workspace
        check(lib.ps_decode(ctypes.byref(self.desc), _vp(q), _vp(pos), hq, ctypes.c_float(scale),
                            _vp(out), _vp(lse), _vp(ws), ws.numel(), _stream(stream)), "ps_decode")
        return out, lse

    def decode_append(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, pos: torch.Tensor,
                      scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      stream=None):
        """ps_decode_append: append one token per sequence (k, v [nseq, Hkv, D] raw at
        pos) and decode q [nseq, Hq, D] at the same positions, in one call."""
        hq = self._check_q(q, pos)
        _shape(k, (self.nseq, self.n_kv_heads, self.head_dim), "k")
        _shape(v, (self.nseq, self.n_kv_heads, self.head_dim), "v")
        if out is not None:
            _shape(out, q.shape, "out")
        if lse is not None:
            _shape(lse, (self.nseq, hq), "lse")
        for t, n in ((q, "q"), (k, "k"), (v, "v")):
            _need(t, BF16, n)
        _need(pos, torch.int32, "pos")
        if scale is None:
            scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(q.shape[0], hq, dtype=torch.float32, device=q.device)
        ws = self.workspace(hq) if workspace is None else workspace
        check(lib.ps_decode_append(ctypes.byref(self.desc), _vp(q), _vp(k), _vp(v), _vp(pos), hq,
                                   ctypes.c_float(scale), _vp(out), _vp(lse), _vp(ws), ws.numel(),
                                   _stream(stream)), "ps_decode_append")
        return out, lse

    def decode_partial(self, q: torch.Tensor, pos: torch.Tensor, scale: Optional[float] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
        """ps_decode_partial: the K/V-streaming launch of ps_decode."""
        hq = self._check_q(q, pos)
        _need(q, BF16, "q")
        _need(pos, torch.int32, "pos")
        if scale is None:
            scale = 1.0 / math.sqrt(self.head_dim)
        ws = self.workspace(hq) if workspace is None else workspace
        check(lib.ps_decode_partial(ctypes.byref(self.desc), _vp(q), _vp(pos), hq,
                                    ctypes.c_float(scale), _vp(ws), ws.numel(), _stream(stream)),
              "ps_decode_partial")

    def decode_combine(self, out: torch.Tensor, lse: torch.Tensor,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
        """ps_decode_combine: merges the partial records into out [nseq,Hq,D] and lse [nseq,Hq]."""
        _dims(out, 3, "out", "[nseq, Hq, D]")
        _shape(out, (self.nseq, out.shape[1], self.head_dim), "out")
        _shape(lse, (self.nseq, out.shape[1]), "lse")
        _need(out, BF16, "out")
        _need(lse, torch.float32, "lse")
        hq = out.shape[1]
        ws = self.workspace(hq) if workspace is None else workspace
        check(lib.ps_decode_combine(ctypes.byref(self.desc), hq, _vp(out), _vp(lse), _vp(ws),
                                    ws.numel(), _stream(stream)), "ps_decode_combine")

    def check_status(self) -> int:
        flags = ctypes.c_int32(0)
        lib.ps_check_device_status(_vp(self.status), ctypes.byref(flags))
        return flags.value


def ring_slots(pos: torch.Tensor, prefix_len: torch.Tensor, window: int, stream=None) -> torch.Tensor:
    _need(pos, torch.int32, "pos")
    _need(prefix_len, torch.int32, "prefix_len")
    out = torch.empty_like(pos)
    check(lib.ps_ring_slots(_vp(pos), _vp(prefix_len), window, _vp(out), pos.numel(),
                            _stream(stream)), "ps_ring_slots")
    return out


def decode_workspace_size(nseq: int, n_q_heads: int, n_kv_heads: int, head_dim: int) -> int:
    b = ctypes.c_size_t(0)
    check(lib.ps_decode_workspace_size(nseq, n_q_heads, n_kv_heads, head_dim, ctypes.byref(b)),
          "ps_decode_workspace_size")
    return b.value


def prefill_workspace_size(batch: int, seqlen: int, n_q_heads: int, n_kv_heads: int,
                           head_dim: int, ring_rows_max: int = 0, pe_mode: int = 0) -> int:
    b = ctypes.c_size_t(0)
    check(lib.ps_prefill_workspace_size(batch, seqlen, n_q_heads, n_kv_heads, head_dim,
                                        ring_rows_max, pe_mode, ctypes.byref(b)),
          "ps_prefill_workspace_size")
    return b.value


def _check_prefill_shapes(q, k, v, q_start, prefix_len):
    _dims(q, 4, "q", "[B, S, Hq, D]")
    _dims(k, 4, "k", "[B, S, Hkv, D]")
    B, S, hq, D = q.shape
    hkv = k.shape[2]
    _shape(k, (B, S, hkv, D), "k")
    _shape(v, (B, S, hkv, D), "v")
    _shape(q_start, (B,), "q_start")
    _shape(prefix_len, (B,), "prefix_len")
    return B, S, hq, D, hkv


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_start: torch.Tensor,
            prefix_len: torch.Tensor, window: int, scale: Optional[float] = None,
            rope_theta: float = 10000.0, ring: Optional[RingCache] = None,
            ring_seq: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            status: Optional[torch.Tensor] = None, stream=None, pe_mode: Optional[int] = None):
    """ps_prefill: q [B,S,Hq,D], k, v [B,S,Hkv,D] bf16 raw.  Returns (out, lse [B,Hq,S]).
    ``pe_mode`` defaults to the ring's (PS_PE_CONTINUE without a ring)."""
    B, S, hq, D, hkv = _check_prefill_shapes(q, k, v, q_start, prefix_len)
    if out is not None:
        _shape(out, q.shape, "out")
    if lse is not None:
        _shape(lse, (B, hq, S), "lse")
    if ring_seq is not None:
        _shape(ring_seq, (B,), "ring_seq")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, BF16, n)
    _need(q_start, torch.int32, "q_start")
    _need(prefix_len, torch.int32, "prefix_len")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, hq, S, dtype=torch.float32, device=q.device)
    ring_rows = 0 if ring is None else ring.prefix_max + ring.window
    if pe_mode is None:
        pe_mode = PS_PE_CONTINUE if ring is None else ring.pe_mode
    if workspace is None:
        workspace = torch.empty(prefill_workspace_size(B, S, hq, hkv, D, ring_rows, pe_mode),
                                dtype=torch.uint8, device=q.device)
    desc = None if ring is None else ctypes.byref(ring.desc)
    check(lib.ps_prefill(_vp(q), _vp(k), _vp(v), B, S, _vp(q_start), _vp(prefix_len), window, hq,
                         hkv, D, ctypes.c_float(scale), ctypes.c_double(rope_theta), pe_mode, desc,
                         _vp(ring_seq), _vp(out), _vp(lse), _vp(workspace), workspace.numel(),
                         _vp(status), _stream(stream)), "ps_prefill")
    return out, lse


def prefill_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                     lse: torch.Tensor, d_out: torch.Tensor, q_start: torch.Tensor,
                     prefix_len: torch.Tensor, window: int, scale: Optional[float] = None,
                     rope_theta: float = 10000.0, status: Optional[torch.Tensor] = None,
                     stream=None, fwd_workspace: Optional[torch.Tensor] = None):
    """ps_prefill_backward: returns fp32 (dq [B,S,Hq,D], dk, dv [B,S,Hkv,D]).
    ``fwd_workspace``: the workspace the forward ps_prefill call (no ring, Continue PE,
    same arguments) used, to reuse its rotated Q and K."""
    B, S, hq, D, hkv = _check_prefill_shapes(q, k, v, q_start, prefix_len)
    _shape(out, q.shape, "out")
    _shape(d_out, q.shape, "d_out")
    _shape(lse, (B, hq, S), "lse")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (d_out, "d_out")):
        _need(t, BF16, n)
    _need(lse, torch.float32, "lse")
    if fwd_workspace is not None:
        need = prefill_workspace_size(B, S, hq, hkv, D)
        if fwd_workspace.numel() < need or not fwd_workspace.is_cuda:
            raise ValueError(f"fwd_workspace: expected a CUDA buffer of at least {need} bytes "
                             "from the forward call")
    _need(q_start, torch.int32, "q_start")
    _need(prefix_len, torch.int32, "prefix_len")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    b = ctypes.c_size_t(0)
    check(lib.ps_prefill_backward_workspace_size(B, S, hq, hkv, D, ctypes.byref(b)),
          "ps_prefill_backward_workspace_size")
    ws = torch.empty(b.value, dtype=torch.uint8, device=q.device)
    check(lib.ps_prefill_backward(_vp(q), _vp(k), _vp(v), _vp(out), _vp(lse), _vp(d_out), B, S,
                                  _vp(q_start), _vp(prefix_len), window, hq, hkv, D,
                                  ctypes.c_float(scale), ctypes.c_double(rope_theta),
                                  _vp(fwd_workspace), _vp(dq), _vp(dk), _vp(dv), _vp(ws), ws.numel(),
                                  _vp(status), _stream(stream)), "ps_prefill_backward")
    return dq, dk, dv


def decode_step_layout(nseq: int, n_q_heads: int, n_kv_heads: int, head_dim: int):
    """ps_decode_step_layout_get: {name: (offset, nbytes)} of the packed input block
    (q, k, v, pos) and of the result block (out, lse), and the blocks' sizes."""
    L = StepLayout()
    check(lib.ps_decode_step_layout_get(nseq, n_q_heads, n_kv_heads, head_dim, ctypes.byref(L)),
          "ps_decode_step_layout_get")
    q_b, kv_b = nseq * n_q_heads * head_dim * 2, nseq * n_kv_heads * head_dim * 2
    inp = {"q": (L.q_off, q_b), "k": (L.k_off, kv_b), "v": (L.v_off, kv_b),
           "pos": (L.pos_off, nseq * 4)}
    res = {"out": (L.out_off, q_b), "lse": (L.lse_off, nseq * n_q_heads * 4)}
    return inp, L.in_bytes, res, L.res_bytes


class DecodeGraph:
    """One decode step of a RingCache (ps_decode_append: one new token per sequence
    appended and attended in one call) captured once in a CUDA graph by the
    library (ps_decode_graph_create) over fixed device buffers.

    The step's inputs live in one packed device buffer ``inp`` (views ``q`` [nseq, Hq,
    D], ``k``, ``v`` [nseq, Hkv, D] bf16 raw, ``pos`` [nseq] int32) and its results in
    one packed buffer ``res`` (views ``out`` [nseq, Hq, D] bf16, ``lse`` [nseq, Hq]
    fp32); ``in_layout`` / ``res_layout`` give (offset, nbytes) of each view, for
    packing host buffers the same way.  ``step(host_in, host_res)`` is one native
    call that copies a packed host input block in, launches the graph, copies the
    results out and waits; ``replay()`` launches the graph alone on inputs already
    in ``inp``.  The object keeps the cache, its workspace and these buffers alive.
    """

    def __init__(self, cache: "RingCache", n_q_heads: int, scale: Optional[float] = None):
        nseq, hkv, D = cache.nseq, cache.n_kv_heads, cache.head_dim
        dev = cache.k_pool.device
        self.in_layout, n_in, self.res_layout, n_res = decode_step_layout(nseq, n_q_heads, hkv, D)
        # 256-byte aligned: torch's caching allocator hands out 512-byte aligned blocks
        self.inp = torch.zeros(n_in, dtype=torch.uint8, device=dev)
        self.res = torch.zeros(n_res, dtype=torch.uint8, device=dev)

        def view(buf, lay, name, dtype, shape):
            o, n = lay[name]
            return buf[o:o + n].view(dtype).view(*shape)

        self.q = view(self.inp, self.in_layout, "q", BF16, (nseq, n_q_heads, D))
        self.k = view(self.inp, self.in_layout, "k", BF16, (nseq, hkv, D))
        self.v = view(self.inp, self.in_layout, "v", BF16, (nseq, hkv, D))
        self.pos = view(self.inp, self.in_layout, "pos", torch.int32, (nseq,))
        self.out = view(self.res, self.res_layout, "out", BF16, (nseq, n_q_heads, D))
        self.lse = view(self.res, self.res_layout, "lse", torch.float32, (nseq, n_q_heads))
        self._ws = torch.empty(decode_workspace_size(nseq, n_q_heads, hkv, D), dtype=torch.uint8,
                               device=dev)
        self.cache = cache
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        self._h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            check(lib.ps_decode_graph_create(ctypes.byref(cache.desc), n_q_heads,
                                             ctypes.c_float(scale), _vp(self.inp), _vp(self.res),
                                             _vp(self._ws), self._ws.numel(),
                                             ctypes.byref(self._h)), "ps_decode_graph_create")

    @staticmethod
    def _host(t: Optional[torch.Tensor], nbytes: int, what: str):
        if t is None:
            return None
        if t.device.type != "cpu" or t.dtype != torch.uint8 or not t.is_contiguous() \
                or t.numel() != nbytes:
            raise ValueError(f"{what}: contiguous uint8 CPU tensor of {nbytes} bytes expected")
        return ctypes.c_void_p(t.data_ptr())

    def step(self, host_in: Optional[torch.Tensor], host_res: Optional[torch.Tensor],
             sync: bool = True, stream=None) -> None:
        """ps_decode_graph_step: copy ``host_in`` (packed like ``inp``; None: ``inp`` is
        already filled) in, run the step, copy the results into ``host_res`` (packed
        like ``res``; None: leave them on the device) and, with ``sync``, wait.  Pinned
        host tensors keep the copies asynchronous."""
        check(lib.ps_decode_graph_step(self._h, self._host(host_in, self.inp.numel(), "host_in"),
                                       self._host(host_res, self.res.numel(), "host_res"),
                                       int(bool(sync)), _stream(stream)), "ps_decode_graph_step")

    def replay(self, stream=None) -> None:
        """Append the step's tokens and decode them (asynchronous; current stream)."""
        self.step(None, None, sync=False, stream=stream)

    def close(self) -> None:
        """Release the graph (steps in flight must have completed)."""
        h, self._h = getattr(self, "_h", None), None
        if h:
            check(lib.ps_decode_graph_destroy(h), "ps_decode_graph_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may be gone
            pass


def prefill_tile_grid(seqlen: int, q_start: int, prefix_len: int, window: int,
                      with_ring: bool = False, bm: int = 128, bn: int = 128):
    nq, nk = ctypes.c_int32(0), ctypes.c_int32(0)
    check(lib.ps_prefill_tile_grid(seqlen, q_start, prefix_len, window, int(with_ring), bm, bn,
                                   ctypes.byref(nq), ctypes.byref(nk)), "ps_prefill_tile_grid")
    return nq.value, nk.value


def prefill_tile_classes(seqlen: int, q_start: int, prefix_len: int, window: int,
                         with_ring: bool = False, bm: int = 128, bn: int = 128,
                         device="cuda", stream=None) -> torch.Tensor:
    nq, nk = prefill_tile_grid(seqlen, q_start, prefix_len, window, with_ring, bm, bn)
    out = torch.empty(nq, nk, dtype=torch.uint8, device=device)
    check(lib.ps_prefill_tile_classes(seqlen, q_start, prefix_len, window, int(with_ring), bm, bn,
                                      _vp(out), _stream(stream)), "ps_prefill_tile_classes")
    return out
