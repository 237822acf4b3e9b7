#!/usr/bin/env python
"""Benchmark of the Prefix-Sliding attention hot path on one B300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

A step is one decode step of one attention layer for a batch of 64 sequences
at position 131,072 (+ step), each with a 64..512-token prefix and a 4,096
window, 16 query / 8 KV heads, head_dim 128: ps_kv_append of the new token's
K/V, then ps_decode (split-KV partial kernel + LSE combine).  `value` is decode
tokens/s for that layer over all ranks.  The same run also measures the
prefill of a 32,768-token sequence (P = 100, W = 4,096) in TFLOP/s, a
full-causal baseline of both from the same library, an end-to-end decode step
through host buffers, and the CPU oracle on the host cores.

Under torchrun (N > 1) every rank runs its own independent batch (replicas,
no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefix-sliding decode tokens/s + HBM GB/s; prefill TFLOP/s vs bf16 peak"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0

# ---- workloads ------------------------------------------------------------
DEC = dict(nseq=64, pos0=131072, W=4096, Pmin=64, Pmax=512, hq=16, hkv=8, D=128, theta=10000.0, seed=3)
PRE = dict(B=1, S=32768, P=100, W=4096, hq=16, hkv=8, D=128, theta=10000.0, seed=2)
LAYERS = 28


def decode_prefix_lens(seed, nseq):
    import synth
    return synth.uniform_int(seed, 10, nseq, DEC["Pmin"], DEC["Pmax"])


def live_runs(p, P, W):
    if p + 1 <= P + W:
        return [(0, p + 1)]
    return ([(0, P)] if P > 0 else []) + [(p - W + 1, W)]


# ---- clocks ---------------------------------------------------------------
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                "clocks.mem")
THROTTLE_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def summarize_clocks(lines):
    """Summary of nvidia-smi samples (CLOCK_FIELDS, csv, no header, no units):
    median SM and memory clocks over the samples drawing at least half the
    peak power (the loaded ones), the highest SM clock limit, and every throttle
    reason seen active under load."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:8],
                         float(parts[8])))
        except ValueError:
            continue
    if not rows:
        return None
    pmax = max(r[2] for r in rows)
    load = [r for r in rows if r[2] >= 0.5 * pmax] or rows
    reasons = sorted({THROTTLE_NAMES[i] for r in load for i, v in enumerate(r[3][1:5])
                      if "Active" in v and "Not" not in v})
    return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
            "mem_mhz": statistics.median(r[4] for r in load), "reasons": reasons,
            "samples": len(rows), "samples_under_load": len(load), "power_w_max": pmax}


class ClockSampler:
    """Samples the GPU's clocks, power and throttle reasons every 100 ms while
    the benchmark runs (nvidia-smi in the background)."""

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        lines = open(self.f.name).read().splitlines()
        os.unlink(self.f.name)
        return summarize_clocks(lines)


# ---- helpers --------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), \
            d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


def committed_traffic(profile: str, source: str):
    """ncu DRAM bytes per launch recorded in a profiles/ summary ("traffic_record:"
    line), if the kernel source still matches the one the counters were taken
    on; else None."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        if line.startswith("traffic_record:"):
            rec = dict(kv.split("=", 1) for kv in line.split(":", 1)[1].split())
    if not rec or rec.get("source") != source:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()
    if rec.get("source_sha256") != sha:
        return None
    return float(rec["dram_bytes_per_launch"])


def fill_random(cache, runs_per_seq, gen, torch, chunk_tokens=1 << 21):
    """Append random raw K/V for each sequence's runs (batched per run index)."""
    depth = max(len(r) for r in runs_per_seq.values())
    dev = cache.k_pool.device
    for i in range(depth):
        items = [(s, r[i]) for s, r in runs_per_seq.items() if i < len(r) and r[i][1] > 0]
        j = 0
        while j < len(items):
            group, tok = [], 0
            while j < len(items) and (not group or tok + items[j][1][1] <= chunk_tokens):
                group.append(items[j])
                tok += items[j][1][1]
                j += 1
            seqs = torch.tensor([s for s, _ in group], dtype=torch.int32, device=dev)
            pos0 = torch.tensor([r[0] for _, r in group], dtype=torch.int32, device=dev)
            cu = torch.tensor(np.concatenate([[0], np.cumsum([r[1] for _, r in group])]),
                              dtype=torch.int32, device=dev)
            shape = (tok, cache.n_kv_heads, cache.head_dim)
            k = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            v = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            cache.append(seqs, pos0, cu, k, v)
            del k, v


# ---- decode ---------------------------------------------------------------
def decode_setup(ps, torch, seed, W, P, pos0, n_steps, full_causal=False, pe_mode=0,
                 block_size=None):
    """Ring cache holding, per sequence, the live K/V of positions < pos0[s]
    (random values), plus every step's q, k, v and positions resident in HBM.
    pos0 is one position for all sequences or one per sequence."""
    d = DEC
    nseq = len(P)
    pos0 = np.broadcast_to(np.asarray(pos0, dtype=np.int64), (nseq,)).copy()
    if full_causal:
        W = int(pos0.max()) + n_steps + 1
        P = np.zeros(nseq, dtype=np.int64)
    prefix_max = int(max(P.max(), d["Pmax"] if not full_causal else 0))
    order = None
    if block_size:  # paged: the sequences' blocks in a shuffled order over the pool
        nblocks = nseq * -(-(prefix_max + W) // block_size)
        order = np.random.default_rng(seed).permutation(nblocks).tolist()
    cache = ps.RingCache(nseq, d["hkv"], d["D"], W, P, rope_theta=d["theta"],
                         prefix_max=prefix_max, zero=False, pe_mode=pe_mode,
                         block_size=block_size, block_order=order)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    runs = {s: live_runs(int(pos0[s]) - 1, int(P[s]), W) for s in range(nseq)}
    fill_random(cache, runs, gen, torch)
    # per-step inputs, resident in HBM before timing
    q = torch.randn(n_steps, nseq, d["hq"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.randn(n_steps, nseq, d["hkv"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(n_steps, nseq, d["hkv"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
    pos = (torch.from_numpy(pos0.astype(np.int32)).cuda()[None, :]
           + torch.arange(n_steps, dtype=torch.int32, device="cuda")[:, None]).contiguous()
    L = np.minimum(pos0 + 1, P + W)  # live slots per sequence once the first step's token is in
    return cache, q, k, v, pos, L


def max_over_ranks(dist, value: float, device: str) -> float:
    """The slowest rank's value (every rank gets it); the value itself without
    a process group.  Replicas run independent batches, so the job's time is the
    slowest replica's."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(base: int, rank: int) -> int:
    """Seed of a replica's synthetic batch: every rank decodes its own sequences."""
    return base + 101 * rank


def job_tokens_per_s(world: int, nseq: int, steps: int, total_ms: float) -> float:
    """Whole-job decode rate: every replica's tokens over the slowest replica's time."""
    return world * nseq * steps / (total_ms / 1e3)


def run_decode(ps, torch, cache, q, k, v, pos, steps, warmup, dist=None, per_kernel=True,
               settle_s=0.0):
    """Times `steps` decode steps (append + partial + combine) after `warmup`.

    The headline loop records no event between the kernels of a step, so
    programmatic dependent launch can overlap their launches; a second pass over
    the same inputs brackets each partial kernel with events for its own time.
    Needs warmup + steps rows of per-step inputs."""
    nseq, hq, D = q.shape[1], q.shape[2], q.shape[3]
    out = torch.empty(nseq, hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(nseq, hq, dtype=torch.float32, device="cuda")
    ws = cache.workspace(hq)
    stream = torch.cuda.current_stream()

    def step(i, evs=None):
        if evs is None:  # the step: ps_decode_append (fused append, partial, combine)
            cache.decode_append(q[i], k[i], v[i], pos[i], out=out, lse=lse, workspace=ws)
            return
        # the same step as three calls, with events around the partial kernel alone
        cache.append_tokens(pos[i], k[i], v[i])
        evs[0].record(stream)
        cache.decode_partial(q[i], pos[i], workspace=ws)
        evs[1].record(stream)
        cache.decode_combine(out, lse, workspace=ws)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    # let the clocks settle under load before timing: repeat the warm-up steps
    # (same positions, same slots) for settle_s seconds
    t_end = time.perf_counter() + settle_s
    while time.perf_counter() < t_end:
        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(dist, e0.elapsed_time(e1), "cuda")
    kern_ms = None
    if per_kernel:
        # the same steps again (the ring's later slots are simply overwritten again):
        # events around each partial kernel, on the stream it runs on
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            step(warmup + i, evs[i])
        torch.cuda.synchronize()
        kern_ms = [a.elapsed_time(b) for a, b in evs]
    return total_ms, kern_ms, out, lse


def decode_leg(ps, torch, name, P, W, pos0, steps, warmup, seed, hbm_peak, pe_mode=0,
               block_size=None):
    """One decode workload: append + partial + combine per step, one layer."""
    d = DEC
    cache, q, k, v, pos, L = decode_setup(ps, torch, seed, W, P, pos0, steps + warmup,
                                          pe_mode=pe_mode, block_size=block_size)
    total_ms, kern_ms, out, _ = run_decode(ps, torch, cache, q, k, v, pos, steps, warmup)
    assert cache.check_status() == 0 and torch.isfinite(out.float()).all()
    nseq = len(P)
    kv = float(np.sum(2 * d["hkv"] * L * d["D"] * 2))
    alg = kv + nseq * d["hq"] * d["D"] * 2
    kern = statistics.mean(kern_ms)
    rep = {"workload": name, "tok_s_per_layer": nseq * steps / (total_ms / 1e3),
           "tok_s_28_layers": nseq * steps / (total_ms / 1e3) / LAYERS,
           "step_ms": total_ms / steps, "partial_kernel_ms": kern,
           "kv_bytes_first_step": kv, "live_slots_mean": float(np.mean(L)),
           "partial_gbs": alg / (kern / 1e3) / 1e9,
           "partial_frac_of_measured_hbm": alg / (kern / 1e3) / 1e9 / hbm_peak}
    del cache, q, k, v, pos
    torch.cuda.empty_cache()
    return rep


def ragged_leg(ps, torch, steps, seed, hbm_peak):
    """256 sequences, positions uniform in [1024, 262143], P in 64..512, W 8,192."""
    import synth
    nseq, W = 256, 8192
    P = synth.uniform_int(seed, 10, nseq, 64, 512)
    pos0 = synth.uniform_int(seed, 11, nseq, 1024, 262143)
    rep = decode_leg(ps, torch, "ragged decode: 256 sequences, positions uniform in [1024, 262143], "
                     "P uniform 64..512, W 8192, Hq 16 / Hkv 8, D 128, one layer", P, W, pos0,
                     steps, 5, seed, hbm_peak)
    rep["sequences_still_causal"] = int(np.sum(pos0 + 1 < P + W))
    return rep


def ragged_full_causal_leg(ps, torch, steps, seed):
    """The ragged decode workload's sequences and positions under full causal
    attention (nothing evicted, every past position cached and read).  Its 143 GB
    of K/V run as two halves of 128 sequences, one after the other; each half's
    cache packs its sequences with per-sequence pool bases (a sequence's rows start
    after the previous sequence's last position), and one step of the whole batch
    is the sum of the two halves' median step times."""
    import synth
    d = DEC
    nseq = 256
    pos0 = synth.uniform_int(seed, 11, nseq, 1024, 262143)  # the ragged leg's draw
    warm = 3
    n_steps = steps + warm
    step_ms, kv_bytes = 0.0, 0.0
    for half in (slice(0, nseq // 2), slice(nseq // 2, nseq)):
        p = pos0[half].astype(np.int64)
        n = len(p)
        W = int(p.max()) + n_steps + 1  # no position ever leaves the window
        used = p + n_steps
        base = np.concatenate([[0], np.cumsum(used)[:-1]])
        cache = ps.RingCache(n, d["hkv"], d["D"], W, np.zeros(n, dtype=np.int64),
                             rope_theta=d["theta"], prefix_max=0, zero=False,
                             slot_base=base.tolist())
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed + 17)
        fill_random(cache, {s: [(0, int(p[s]))] for s in range(n)}, gen, torch)
        shape = (n_steps, n)
        q = torch.randn(*shape, d["hq"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
        k = torch.randn(*shape, d["hkv"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
        v = torch.randn(*shape, d["hkv"], d["D"], generator=gen, device="cuda").to(torch.bfloat16)
        pos = (torch.from_numpy(p.astype(np.int32)).cuda()[None, :]
               + torch.arange(n_steps, dtype=torch.int32, device="cuda")[:, None]).contiguous()
        step_ms += statistics.median(step_times(ps, torch, cache, q, k, v, pos, steps, warm))
        kv_bytes += float(np.sum(2 * d["hkv"] * (p + 1) * d["D"] * 2))
        del cache, q, k, v, pos
        torch.cuda.empty_cache()
    return {"decode_tok_s": nseq / (step_ms / 1e3), "decode_ms_per_step": step_ms,
            "kv_gb_per_step": kv_bytes / 1e9,
            "how": "same library and sequences, W > every position (no eviction), P = 0; two "
                   "halves of 128 sequences run one after the other (%.0f GB of K/V read per "
                   "step in all), step time = sum of the halves' medians over %d steps"
                   % (kv_bytes / 1e9, steps)}


def step_times(ps, torch, cache, q, k, v, pos, steps, warmup):
    """Per-step device times (ms) of `steps` decode steps (append + partial +
    combine), each bracketed by events on the launching stream, after `warmup`."""
    nseq, hq, D = q.shape[1], q.shape[2], q.shape[3]
    out = torch.empty(nseq, hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(nseq, hq, dtype=torch.float32, device="cuda")
    ws = cache.workspace(hq)
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        cache.append_tokens(pos[i], k[i], v[i])
        cache.decode(q[i], pos[i], out=out, lse=lse, workspace=ws)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        cache.append_tokens(pos[warmup + i], k[warmup + i], v[warmup + i])
        cache.decode(q[warmup + i], pos[warmup + i], out=out, lse=lse, workspace=ws)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    assert cache.check_status() == 0 and torch.isfinite(out.float()).all()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def flatness_leg(ps, torch, seed, steps=200, rounds=2):
    """Steady-decode shapes at growing positions: cost must stop growing once
    every sequence's window is full (p >= P + W - 1).  Each position is measured
    `rounds` times in a shuffled order (a fresh cache each time), `steps` steps
    each; per position the median and minimum step time over all its steps."""
    d = DEC
    P = decode_prefix_lens(seed, d["nseq"])
    W = d["W"]
    labels = (("P+W/2", P + W // 2), ("P+W", P + W), ("2(P+W)", 2 * (P + W)),
              ("32768", np.full(d["nseq"], 32768)), ("131072", np.full(d["nseq"], 131072)),
              ("262143", np.full(d["nseq"], 262143 - steps - 8)))
    order = [i for _ in range(rounds) for i in range(len(labels))]
    np.random.default_rng(seed).shuffle(order)
    times = {i: [] for i in range(len(labels))}
    live = {}
    for i in order:
        label, pos0 = labels[i]
        cache, q, k, v, pos, L = decode_setup(ps, torch, seed + 31 * i, W, P, pos0, steps + 5)
        times[i].append(step_times(ps, torch, cache, q, k, v, pos, steps, 5))
        live[i] = float(np.mean(L))
        del cache, q, k, v, pos
        torch.cuda.empty_cache()
    out = []
    for i, (label, _) in enumerate(labels):
        allt = [t for run in times[i] for t in run]
        out.append({"p": label, "live_slots_mean": live[i], "step_ms_median": statistics.median(allt),
                    "step_ms_min": min(allt),
                    "step_ms_median_per_round": [statistics.median(r) for r in times[i]],
                    "tok_s_per_layer": d["nseq"] / (statistics.median(allt) / 1e3)})
    full = [o["step_ms_median"] for o in out if o["p"] != "P+W/2"]
    return {"positions": out, "steps_per_round": steps, "rounds": rounds, "order": order,
            "max_over_min_median_full_window": max(full) / min(full)}


def small_batch_leg(ps, torch, seed, steps=200):
    """Decode latency of one sequence (16 / 8 heads, D 128, P 100, W 4,096) at
    p = 1,000 (still causal) and p = P + W (window full): one step (append +
    partial + combine) replayed `steps` times back to back from a CUDA graph
    (DecodeGraph, the serving path; the step's position stays fixed, so each
    replay rewrites the same slot), and the same step launched eagerly through
    the Python binding, whose host work then sets the pace."""
    out = {}
    P = np.array([100])
    for label, p0 in (("p=1000", 1000), ("p=P+W", 100 + 4096)):
        cache, q, k, v, pos, L = decode_setup(ps, torch, seed, 4096, P, p0, steps + 5)
        eager = step_times(ps, torch, cache, q, k, v, pos, steps, 5)
        g = ps.DecodeGraph(cache, DEC["hq"])
        g.q.copy_(q[0])
        g.k.copy_(k[0])
        g.v.copy_(v[0])
        g.pos.copy_(pos[0])
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        assert cache.check_status() == 0 and torch.isfinite(g.out.float()).all()
        out[label] = {"graph_step_us": 1e3 * e0.elapsed_time(e1) / steps,
                      "eager_step_us_median": 1e3 * statistics.median(eager),
                      "live_slots": int(L[0])}
        del g, cache, q, k, v, pos
        torch.cuda.empty_cache()
    return out


def comparator_legs(ps, torch, args, seed, hbm_peak, bf16_peak):
    """The same library on the same shapes with a plain sliding window (P = 0)
    and a StreamingLLM-style 4-token sink (P = 4): decode at the steady-decode
    shapes, prefill at the 32K prefill shape; Reset PE decode and prefill at
    those shapes; and decode through a paged ring (shuffled 64-slot blocks)."""
    d = DEC
    out = {}
    for name, pval in (("sliding_window_P0", 0), ("streaming_sink_P4", 4)):
        P = np.full(d["nseq"], pval, dtype=np.int64)
        r = decode_leg(ps, torch, f"decode, 64 x 131072, W 4096, P = {pval}", P, d["W"], d["pos0"],
                       100, 5, seed + 11, hbm_peak)
        rep = {"decode_tok_s_per_layer": r["tok_s_per_layer"], "decode_step_ms": r["step_ms"],
               "decode_partial_ms": r["partial_kernel_ms"], "decode_partial_gbs": r["partial_gbs"]}
        if not args.no_prefill:
            pr = prefill_report(ps, torch, f"prefill 32768, W 4096, P = {pval}", 1, PRE["S"], pval,
                                PRE["W"], args.prefill_steps, seed + 12, bf16_peak)
            rep.update({"prefill_ms": pr["ms"], "prefill_tflops_algorithmic": pr["tflops_algorithmic"],
                        "prefill_frac_of_measured_bf16": pr["frac_of_measured_bf16_burst"]})
        out[name] = rep
    # Reset PE: the same steady-decode shapes with the cache renumbered per query
    P = decode_prefix_lens(seed, d["nseq"])
    r = decode_leg(ps, torch, "decode, 64 x 131072, W 4096, Reset PE", P, d["W"], d["pos0"], 100, 5,
                   seed + 13, hbm_peak, pe_mode=ps.PS_PE_RESET)
    out["reset_pe"] = {"decode_tok_s_per_layer": r["tok_s_per_layer"], "decode_step_ms": r["step_ms"],
                       "decode_partial_ms": r["partial_kernel_ms"], "decode_partial_gbs": r["partial_gbs"],
                       "decode_partial_frac_of_measured_hbm": r["partial_frac_of_measured_hbm"]}
    # Reset PE prefill at the 32K shape (prefix tiles visited with the renumbered query)
    if not args.no_prefill:
        try:
            ms, _ = run_prefill(ps, torch, PRE["S"], PRE["P"], PRE["W"], args.prefill_steps, 3,
                                seed + 14, pe_mode=ps.PS_PE_RESET)
            flops = prefill_flops(PRE["S"], PRE["P"], PRE["W"], PRE["hq"], PRE["D"])
            out["reset_pe"].update({"prefill_ms": ms, "prefill_tflops_algorithmic": flops / ms / 1e9})
        except Exception as e:  # a comparator must not take the bench line down
            out["reset_pe"]["prefill_error"] = str(e)[:200]
    # paged ring (64-slot blocks in a shuffled order) at the steady-decode shapes
    try:
        r = decode_leg(ps, torch, "decode, 64 x 131072, W 4096, paged (64-slot blocks, shuffled)",
                       decode_prefix_lens(seed, d["nseq"]), d["W"], d["pos0"], 100, 5, seed + 15,
                       hbm_peak, block_size=64)
        out["paged_block64"] = {"decode_tok_s_per_layer": r["tok_s_per_layer"],
                                "decode_step_ms": r["step_ms"],
                                "decode_partial_ms": r["partial_kernel_ms"],
                                "decode_partial_gbs": r["partial_gbs"],
                                "decode_partial_frac_of_measured_hbm": r["partial_frac_of_measured_hbm"]}
    except Exception as e:
        out["paged_block64"] = {"error": str(e)[:200]}
    return out


def run_decode_e2e(ps, torch, cache, steps, warmup, seed):
    """Same decode step through host buffers, with the package's DecodeGraph: per
    step one native call (ps_decode_graph_step) that issues the pinned host ->
    device copy of the step's packed q, k, v, pos, the graph launch (append +
    decode) and the device -> host copy of the packed O and LSE, then waits for
    the stream.  Each timed step reads its own host input row."""
    d = DEC
    nseq, hq, hkv, D = d["nseq"], d["hq"], d["hkv"], d["D"]
    g = ps.DecodeGraph(cache, hq)
    n = steps + warmup
    gen = torch.Generator().manual_seed(seed)
    hin = torch.zeros(n, g.inp.numel(), dtype=torch.uint8).pin_memory()
    for name, heads in (("q", hq), ("k", hkv), ("v", hkv)):
        o, nb = g.in_layout[name]
        hin[:, o:o + nb].view(torch.bfloat16).view(n, nseq, heads, D).copy_(
            torch.randn(n, nseq, heads, D, generator=gen).to(torch.bfloat16))
    start = d["pos0"] + 100000  # positions after the device-resident run
    o, nb = g.in_layout["pos"]
    hin[:, o:o + nb].view(torch.int32).copy_(
        (start + torch.arange(n, dtype=torch.int32))[:, None].repeat(1, nseq))
    hres = torch.empty(g.res.numel(), dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream()

    for i in range(warmup):
        g.step(hin[i], hres)
    t0 = time.perf_counter()
    for i in range(steps):
        g.step(hin[warmup + i], hres)
    dt = time.perf_counter() - t0

    # where a step goes: the host wall clock of the same native call with the
    # copies left out one at a time (re-appending the last rows' positions), and
    # the graph's device time between events
    def wall(fn):
        ts = []
        for i in range(steps):
            h0 = time.perf_counter()
            fn(warmup + i)
            ts.append(1e3 * (time.perf_counter() - h0))
        return statistics.median(ts)

    parts = {"step_ms": wall(lambda i: g.step(hin[i], hres)),
             "without_d2h_ms": wall(lambda i: g.step(hin[i], None)),
             "without_h2d_ms": wall(lambda i: g.step(None, hres)),
             "graph_only_ms": wall(lambda i: g.step(None, None))}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dev = []
    for _ in range(steps):
        e0.record(stream)
        g.replay()
        e1.record(stream)
        stream.synchronize()
        dev.append(e0.elapsed_time(e1))
    parts["graph_device_ms"] = statistics.median(dev)
    parts["h2d_cost_ms"] = parts["step_ms"] - parts["without_h2d_ms"]
    parts["d2h_cost_ms"] = parts["step_ms"] - parts["without_d2h_ms"]
    parts["launch_and_sync_ms"] = parts["graph_only_ms"] - parts["graph_device_ms"]
    g.close()
    return dt, g.inp.numel(), g.res.numel(), parts


# ---- prefill --------------------------------------------------------------
def prefill_flops(S, P, W, hq, D, bm=128, bn=128):
    """Exact admitted (query, key) pairs and the pairs inside non-skipped tiles."""
    p = np.arange(S, dtype=np.int64)
    pairs = np.minimum(p + 1, P + W).sum()
    return 4.0 * D * hq * float(pairs)


def timed_rounds(torch, fn, steps, rounds=5):
    """Device time per call of fn(): `rounds` rounds of about steps / rounds calls,
    each round between CUDA events with a synchronisation on both sides; returns
    the median over rounds of the per-call mean, and the per-round means (a
    transient clock drop from the power cap moves one round, not the median)."""
    per = max(1, -(-steps // rounds))
    means = []
    for _ in range(rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(per):
            fn()
        e1.record()
        torch.cuda.synchronize()
        means.append(e0.elapsed_time(e1) / per)
    return statistics.median(means), means


def run_prefill(ps, torch, S, P, W, steps, warmup, seed, full_causal=False, B=None, pe_mode=0):
    """Times whole ps_prefill calls (RoPE pre-pass + tile kernel) on one layer's
    resident q, k, v; returns ms per call and the tile classes of one row."""
    d = PRE
    B = d["B"] if B is None else B
    hq, hkv, D = d["hq"], d["hkv"], d["D"]
    if full_causal:
        W = S
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    q = torch.randn(B, S, hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, S, hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, S, hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    qs = torch.zeros(B, dtype=torch.int32, device="cuda")
    pl = torch.full((B,), P, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, hq, S, dtype=torch.float32, device="cuda")
    ws = torch.empty(ps.prefill_workspace_size(B, S, hq, hkv, D, pe_mode=pe_mode),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(warmup):
        ps.prefill(q, k, v, qs, pl, W, rope_theta=d["theta"], out=out, lse=lse, workspace=ws,
                   status=status, pe_mode=pe_mode)
    ms, _ = timed_rounds(torch, lambda: ps.prefill(q, k, v, qs, pl, W, rope_theta=d["theta"],
                                                   out=out, lse=lse, workspace=ws, status=status,
                                                   pe_mode=pe_mode),
                         steps)
    assert int(status.item()) == 0, f"prefill device status {int(status.item())}"
    assert torch.isfinite(lse).all()
    cls = ps.prefill_tile_classes(S, 0, P, W).cpu().numpy()
    n_skip, n_part, n_full = [(cls == c).sum() for c in (0, 1, 2)]
    return ms, dict(skip=int(n_skip), partial=int(n_part), full=int(n_full))


def prefill_report(ps, torch, name, B, S, P, W, steps, seed, bf16_peak, full_causal_steps=0):
    """Prefill leg: algorithmic and executed TFLOP/s of one ps_prefill call."""
    d = PRE
    ms, cls = run_prefill(ps, torch, S, P, W, steps, 3, seed, B=B)
    flops = B * prefill_flops(S, P, W, d["hq"], d["D"])
    tile_flops = B * 4.0 * d["D"] * d["hq"] * 128 * 128 * (cls["partial"] + cls["full"])
    nq = -(-S // 128)
    causal_tiles = nq * (nq + 1) // 2
    rep = {"workload": name, "ms": ms, "tflops_algorithmic": flops / ms / 1e9,
           "tflops_on_nonskipped_tiles": tile_flops / ms / 1e9,
           "frac_of_measured_bf16_burst": tile_flops / ms / 1e9 / bf16_peak,
           "timed": "whole ps_prefill call: RoPE pre-pass + tile kernel; median over 5 rounds "
                    "of the per-call mean",
           "tiles_per_row_and_head": cls,
           "skip_fraction_of_causal_tiles": 1 - (cls["partial"] + cls["full"]) / causal_tiles}
    if full_causal_steps:
        fms, _ = run_prefill(ps, torch, S, 0, W, full_causal_steps, 2, seed + 9, full_causal=True, B=B)
        rep["full_causal_ms"] = fms
        rep["speedup_vs_full_causal"] = fms / ms
    torch.cuda.empty_cache()
    return rep


def backward_report(ps, torch, B, S, P, W, steps, seed, bf16_peak):
    """Training backward (dq, dk, dv) of the truncated-backprop step, one layer."""
    d = PRE
    hq, hkv, D = d["hq"], d["hkv"], d["D"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    q = torch.randn(B, S, hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, S, hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, S, hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    do = torch.randn(B, S, hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    qs = torch.zeros(B, dtype=torch.int32, device="cuda")
    pl = torch.full((B,), P, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the forward's workspace keeps its rotated Q and K, which the backward reuses
    fws = torch.empty(ps.prefill_workspace_size(B, S, hq, hkv, D), dtype=torch.uint8, device="cuda")
    out, lse = ps.prefill(q, k, v, qs, pl, W, rope_theta=d["theta"], workspace=fws, status=status)
    for _ in range(2):
        ps.prefill_backward(q, k, v, out, lse, do, qs, pl, W, rope_theta=d["theta"], status=status,
                            fwd_workspace=fws)
    ms, _ = timed_rounds(torch, lambda: ps.prefill_backward(
        q, k, v, out, lse, do, qs, pl, W, rope_theta=d["theta"], status=status,
        fwd_workspace=fws), steps)
    assert int(status.item()) == 0
    fwd_alg = B * prefill_flops(S, P, W, hq, D)
    exe = B * backward_executed_flops(S, P, W, hq, hkv, D)
    torch.cuda.empty_cache()
    return {"workload": f"training backward {B} x {S}, P={P}, W={W}, Hq 16 / Hkv 8, D 128, one layer",
            "ms": ms, "tflops_algorithmic": 2.5 * fwd_alg / ms / 1e9,
            "tflops_executed": exe / ms / 1e9,
            "frac_of_measured_bf16_burst": 2.5 * fwd_alg / ms / 1e9 / bf16_peak,
            "timed": "median over 5 rounds of the per-call mean of whole ps_prefill_backward "
                     "calls reusing the forward's rotated Q and K: "
                     "pre-pass (D = rowsum(dO * O)) + the dQ / dK,dV kernel; "
                     "algorithmic = 2.5 x forward FLOPs (dV, dP, dQ, dK over the admitted pairs), "
                     "executed = the tensor-core products the kernels issue"}


def backward_executed_flops(S, P, W, hq, hkv, D, c0=0):
    """FLOPs of the tensor-core products the backward issues for one batch row:
    each dQ CTA (128 queries) runs S, dP and dQ over the forward's 128-key
    tiles, each dK/dV CTA (128 keys) runs S, dP, dV and dK over the 128-query
    tiles that can see its keys, for every query head of its group."""
    def cdiv(a, b):
        return -(-a // b)

    def clamp(x):
        return max(0, min(S, x))

    tile = 2.0 * 128 * 128 * D
    n_dq = n_kv = 0
    nq = cdiv(S, 128)
    for t in range(nq):
        r0, r1 = t * 128, min(S, t * 128 + 128) - 1
        kc, kp = clamp(r1 + 1), clamp(P - c0)
        t1 = cdiv(min(kp, kc), 128)
        t2b = max(t1, clamp(r0 - W + 1) // 128)
        n_dq += t1 + max(0, cdiv(kc, 128) - t2b)
        qe = nq if c0 + r0 < P else min(nq, (r1 + W - 1) // 128 + 1)
        n_kv += max(0, qe - t)
    return tile * (3 * hq * n_dq + 4 * hq * n_kv)


# ---- CPU oracle -----------------------------------------------------------
def _oracle_worker(args):
    """Spawned worker: builds one sequence's visible history (untimed), then
    times the oracle's attention for the query."""
    seq, pos, P, W, hq, hkv, D, theta, seed = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np_  # noqa: F401
    import synth
    from oracle import attend, visible_positions
    hist = synth.History(seed, seq, hkv, D)
    js = visible_positions(pos, P, W)
    k, v = hist.rows(js)
    lut = {int(j): i for i, j in enumerate(js)}

    def history(req):
        idx = [lut[int(j)] for j in req]
        return k[idx], v[idx]

    q = synth.bits_to_f64(synth.query_bits(seed, seq, pos, hq, D))[0]
    t0 = time.perf_counter()
    attend(q, pos, P, W, history, theta)
    return time.perf_counter() - t0


def oracle_baseline(budget_s=20.0):
    """Oracle decode throughput on this host's cores over a bounded sample of
    the decode workload (tokens/s for one layer)."""
    import multiprocessing as mp
    d = DEC
    P = decode_prefix_lens(d["seed"], d["nseq"])
    cores = max(1, min(os.cpu_count() or 1, 32))
    jobs = [(s % d["nseq"], d["pos0"], int(P[s % d["nseq"]]), d["W"], d["hq"], d["hkv"], d["D"],
             d["theta"], d["seed"]) for s in range(d["nseq"])]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        times = pool.map(_oracle_worker, jobs[:cores])   # calibrate
        per_seq = statistics.median(times)
        n = int(max(cores, min(len(jobs) * 8, budget_s * cores / max(per_seq, 1e-3))))
        work = [jobs[i % len(jobs)] for i in range(n)]
        t1 = time.perf_counter()
        times = pool.map(_oracle_worker, work, chunksize=1)
        wall = time.perf_counter() - t1
    busy = sum(times)
    # throughput of the attention compute: sequences done per second of the
    # cores' attention time (history generation excluded)
    value = n / (busy / cores)
    return {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} decode queries (all 16 heads each) of the steady-decode workload, "
                      f"float64 numpy oracle, {cores} spawned processes, attention time only "
                      f"(history synthesis excluded); wall {wall:.1f} s",
            "cpu_seconds": busy}


def oracle_prefill_baseline(budget_s=10.0):
    """Oracle prefill throughput on this host's cores over a bounded sample of
    the 32K-prefill workload: query rows past the first full window (each
    attends P + W keys, as most rows of the prompt do), all 16 heads each,
    history synthesis excluded.  Rows per second of one layer."""
    import multiprocessing as mp
    d = PRE
    cores = max(1, min(os.cpu_count() or 1, 32))
    rows = list(range(d["P"] + d["W"], d["S"], 97))  # a spread of steady rows
    jobs = [(0, r, d["P"], d["W"], d["hq"], d["hkv"], d["D"], d["theta"], 17) for r in rows]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        times = pool.map(_oracle_worker, jobs[:cores])   # calibrate
        per_row = statistics.median(times)
        n = int(max(cores, min(len(jobs), budget_s * cores / max(per_row, 1e-3))))
        t1 = time.perf_counter()
        times = pool.map(_oracle_worker, jobs[:n], chunksize=1)
        wall = time.perf_counter() - t1
    busy = sum(times)
    return {"value": n / (busy / cores), "unit": "query rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} query rows (positions {d['P'] + d['W']}..{d['S'] - 1}, step 97, all 16 "
                      f"heads each) of the 32K prefill, float64 numpy oracle, {cores} spawned "
                      f"processes, attention time only; wall {wall:.1f} s",
            "cpu_seconds": busy}


# ---- main -----------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-baselines", action="store_true", help="skip full-causal and oracle legs")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the ragged-decode and flatness legs")
    ap.add_argument("--only", choices=["prefill", "train", "backward"],
                    help="run one prefill leg alone (--prefill-steps timed calls, few launches "
                         "before them) and print its report instead of the contract line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist_
        torch.cuda.set_device(local)
        dist_.init_process_group("nccl")
        dist = dist_
    else:
        torch.cuda.set_device(0)
    import prefix_sliding_window_02_b300 as ps

    hbm_peak, bf16_peak, _, peak_src = peaks()
    if args.only:
        return only_leg(ps, torch, args, bf16_peak)
    d = DEC
    seed = replica_seed(d["seed"], rank)
    P = decode_prefix_lens(seed, d["nseq"])
    n_steps = args.warmup + args.steps
    cache, q, k, v, pos, L = decode_setup(ps, torch, seed, d["W"], P, d["pos0"], n_steps)
    clocks = ClockSampler(local)
    total_ms, kern_ms, out, _ = run_decode(ps, torch, cache, q, k, v, pos, args.steps, args.warmup, dist,
                                           settle_s=0.5)
    assert cache.check_status() == 0
    assert torch.isfinite(out.float()).all()
    ms_step = total_ms / args.steps
    value = job_tokens_per_s(world, d["nseq"], args.steps, total_ms)

    kv_bytes = float(np.sum(2 * d["hkv"] * L * d["D"] * 2))  # K and V of the live slots
    q_bytes = d["nseq"] * d["hq"] * d["D"] * 2
    alg_bytes = kv_bytes + q_bytes
    kern_avg_ms = statistics.mean(kern_ms)
    achieved = alg_bytes / (kern_avg_ms / 1e3) / 1e9
    step_gbs = alg_bytes / (ms_step / 1e3) / 1e9

    e2e = None
    full = None
    pre = None
    if rank == 0 or world == 1:
        e2e_steps = 200
        dt, h2d, d2h, parts = run_decode_e2e(ps, torch, cache, e2e_steps, 10, seed + 7)
        e2e = {"value": d["nseq"] * e2e_steps / dt, "unit": "tok/s", "steps": e2e_steps,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "breakdown_median": parts,
               "how": "per step one native call (DecodeGraph.step -> ps_decode_graph_step): "
                      "pinned host -> device copy of the packed q, k, v, pos; launch of "
                      "ps_decode_append captured in a CUDA graph; device -> host copy of the "
                      "packed O and LSE; stream sync; host wall clock over 200 steps. "
                      "breakdown_median: host wall clock of one such call, and with either "
                      "copy left out; graph_device_ms: the graph between CUDA events"}
    del cache, q, k, v
    torch.cuda.empty_cache()

    # the other decode legs run before the prefill legs, whose power draw can
    # leave the next few hundred milliseconds of decode slower
    ragged = flat = comparators = small = None
    if not args.no_extra and (rank == 0 or world == 1):
        ragged = ragged_leg(ps, torch, 100, 4, hbm_peak)
        flat = flatness_leg(ps, torch, seed)
        small = small_batch_leg(ps, torch, seed + 21)
        comparators = comparator_legs(ps, torch, args, seed, hbm_peak, bf16_peak)
        # last of the decode legs: its 135 GB-per-step run draws the most power
        if not args.no_baselines:
            fc = ragged_full_causal_leg(ps, torch, 10, 4)
            fc["decode_speedup"] = fc["decode_ms_per_step"] / ragged["step_ms"]
            ragged["full_causal"] = fc

    # prefill (one layer) and the truncated-backprop training forward
    try:
        if args.no_prefill:
            raise RuntimeError("prefill leg skipped (--no-prefill)")
        fc = 0 if args.no_baselines else 3
        pre = prefill_report(ps, torch, "prefill 1 x 32768 tokens, P=100, W=4096, Hq 16 / Hkv 8, "
                             "D 128, one layer", 1, PRE["S"], PRE["P"], PRE["W"], args.prefill_steps,
                             seed + 5, bf16_peak, fc)
        train = prefill_report(ps, torch, "training forward 8 x 8192 tokens, P=256, W=2048, Hq 16 / "
                               "Hkv 8, D 128, one layer", 8, 8192, 256, 2048, args.prefill_steps,
                               seed + 6, bf16_peak, fc)
        train["backward"] = backward_report(ps, torch, 8, 8192, 256, 2048, max(3, args.prefill_steps // 2),
                                            seed + 8, bf16_peak)
    except Exception as e:  # noqa: BLE001
        pre = {"unavailable": f"{type(e).__name__}: {e}"}
        train = None

    if not args.no_baselines and (rank == 0 or world == 1):
        fsteps = min(args.steps, 30)
        cfc, qf, kf, vf, posf, Lf = decode_setup(ps, torch, seed + 3, d["W"], P, d["pos0"],
                                                 fsteps + 3, full_causal=True)
        fms, _, _, _ = run_decode(ps, torch, cfc, qf, kf, vf, posf, fsteps, 3, None, per_kernel=False)
        full = {"decode_tok_s": d["nseq"] * fsteps / (fms / 1e3), "decode_ms_per_step": fms / fsteps,
                "kv_gb_per_step": float(np.sum(2 * d["hkv"] * Lf * d["D"] * 2)) / 1e9,
                "how": "same library, W > position (no eviction), P = 0"}
        del cfc, qf, kf, vf
        torch.cuda.empty_cache()
        full["decode_speedup"] = value / world / full["decode_tok_s"]
    clk = clocks.stop()

    cpu = None
    if not args.no_baselines and world == 1:
        cpu = oracle_baseline()
        if pre is not None and "ms" in pre:
            pre["cpu_baseline"] = oracle_prefill_baseline()
            pre["gpu_query_rows_per_s"] = PRE["S"] / (pre["ms"] / 1e3)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (N(0,1) bf16 K/V/Q, random-init)",
        "config": {"workload": "steady decode: 64 sequences at position 131072+step, P uniform "
                               "64..512, W 4096, Hq 16 / Hkv 8, D 128, one layer per step "
                               "(ps_decode_append: the new token's append inside the split-KV "
                               "partial kernel, then the combine)",
                   "layers_for_model_rate": LAYERS, "l2": "inputs larger than L2 "
                   f"({kv_bytes / 1e9:.2f} GB of K/V read per step vs 126 MB L2)",
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "decode": {"tok_s_per_layer": value, "tok_s_28_layers": value / LAYERS,
                   "step_hbm_gbs": step_gbs, "kv_bytes_per_step": kv_bytes,
                   "partial_kernel_ms": kern_avg_ms, "step_ms": ms_step},
        "roofline": {"kernel": "decode_partial_kernel<128,2,8,3,false>", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_src} hbm_gbs",
                     "traffic": committed_traffic("decode_partial_steady_64x131072.md",
                                                  "prefix_sliding_window_02_b300/csrc/ps_decode.cu"),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "frac_of_8tbs": achieved / 8000.0},
        "prefill": pre, "train_forward": train, "ragged_decode": ragged, "flatness": flat,
        "small_batch_decode": small,
        "comparators": comparators,
        "full_causal": full, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clk, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def only_leg(ps, torch, args, bf16_peak):
    """One prefill leg by itself, e.g. as the program a profiler captures."""
    n = args.prefill_steps
    if args.only == "prefill":
        r = prefill_report(ps, torch, "prefill 1 x 32768 tokens, P=100, W=4096, Hq 16 / Hkv 8, "
                           "D 128, one layer", 1, PRE["S"], PRE["P"], PRE["W"], n, 17, bf16_peak, 0)
    elif args.only == "train":
        r = prefill_report(ps, torch, "training forward 8 x 8192 tokens, P=256, W=2048, Hq 16 / "
                           "Hkv 8, D 128, one layer", 8, 8192, 256, 2048, n, 18, bf16_peak, 0)
    else:
        r = backward_report(ps, torch, 8, 8192, 256, 2048, n, 20, bf16_peak)
    print(json.dumps({"leg": args.only, **r}), flush=True)


def reference_arm(args, world, rank):
    """The oracle as the reference arm: timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    t0 = time.perf_counter()
    runs = []
    for _ in range(args.warmup + args.steps):
        runs.append(oracle_baseline(budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup))))
    timed = runs[args.warmup:]
    value = statistics.mean(r["value"] for r in timed)
    cpu = dict(timed[-1])
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * DEC["nseq"] / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "steady decode: 64 sequences at position 131072, P uniform 64..512, "
                                   "W 4096, Hq 16 / Hkv 8, D 128, one layer (bounded sample per step)"},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
