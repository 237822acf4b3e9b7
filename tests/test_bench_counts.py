"""The work counts bench.py divides by (no GPU): the prefill's algorithmic FLOPs
come from the exact number of admitted (query, key) pairs, and the backward's
issued products cover every tile pair the mask reaches."""
import os
import sys

import numpy as np
import pytest

from oracle import allowed, tile_classes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("S", [1, 7, 40])
def test_prefill_flops_counts_admitted_pairs(S):
    for P in range(0, S + 2, 3):
        for W in range(1, S + 3, 4):
            pairs = sum(allowed(p, j, P, W) for p in range(S) for j in range(S))
            assert bench.prefill_flops(S, P, W, 1, 1) == 4.0 * pairs, (S, P, W)


@pytest.mark.parametrize("S,P,W", [(1000, 100, 256), (700, 0, 128), (513, 600, 64), (2048, 256, 512)])
def test_backward_products_cover_every_reached_tile(S, P, W):
    """Each non-skipped 128 x 128 tile pair is visited by one dQ CTA (3 products)
    and, for each query head, by one dK/dV CTA (4 products): at least 7 tile
    products per non-skipped tile and head."""
    pos = np.arange(S)
    cls = tile_classes(pos, pos, P, W, 128, 128)
    reached = int((np.asarray(cls) > 0).sum())
    tile = 2.0 * 128 * 128 * 128
    issued = bench.backward_executed_flops(S, P, W, hq=1, hkv=1, D=128)
    assert issued >= 7 * tile * reached
    # and it visits nothing beyond the forward's tile ranges: at most the causal triangle
    nq = -(-S // 128)
    assert issued <= 7 * tile * nq * (nq + 1) // 2


def test_clock_summary_reads_loaded_samples_and_reasons():
    idle = "345, 2032, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 3996"
    busy = "2032, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active, 3996"
    slow = "1500, 2032, 880.0, 0x8, Active, Not Active, Not Active, Not Active, 3996"
    r = bench.summarize_clocks([idle, busy, busy, slow, "garbage", ""])
    assert r["samples"] == 4 and r["samples_under_load"] == 3
    assert r["sm_mhz"] == 2032 and r["sm_max_mhz"] == 2032 and r["mem_mhz"] == 3996
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.summarize_clocks(["x"]) is None
