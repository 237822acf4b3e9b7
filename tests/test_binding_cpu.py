"""The Python binding checks every tensor's shape before a pointer reaches the
library (which trusts the sizes it is given); these checks run before any
device check, so they are exercised here with CPU tensors."""
import pytest
import torch


@pytest.fixture(scope="module")
def ps():
    import prefix_sliding_window_02_b300 as ps
    return ps


def _inputs(B=2, S=5, hq=4, hkv=2, D=128):
    bf = torch.bfloat16
    return (torch.zeros(B, S, hq, D, dtype=bf), torch.zeros(B, S, hkv, D, dtype=bf),
            torch.zeros(B, S, hkv, D, dtype=bf), torch.zeros(B, dtype=torch.int32),
            torch.zeros(B, dtype=torch.int32))


@pytest.mark.parametrize("bad, what", [
    ("k", "k"), ("v", "v"), ("q_start", "q_start"), ("prefix_len", "prefix_len"),
])
def test_prefill_rejects_mismatched_shapes(ps, bad, what):
    q, k, v, qs, pl = _inputs()
    args = dict(k=k, v=v, q_start=qs, prefix_len=pl)
    t = args[bad]
    args[bad] = t[:1] if t.dim() == 1 else t[:, :3]
    with pytest.raises(ValueError, match=what):
        ps.prefill(q, args["k"], args["v"], args["q_start"], args["prefix_len"], 16)


def test_prefill_rejects_bad_out_lse_and_ranks(ps):
    q, k, v, qs, pl = _inputs()
    with pytest.raises(ValueError, match="out"):
        ps.prefill(q, k, v, qs, pl, 16, out=torch.zeros(2, 5, 4, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="lse"):
        ps.prefill(q, k, v, qs, pl, 16, lse=torch.zeros(2, 5, 4))  # must be [B, Hq, S]
    with pytest.raises(ValueError, match="q"):
        ps.prefill(q[0], k, v, qs, pl, 16)


def test_backward_rejects_mismatched_shapes(ps):
    q, k, v, qs, pl = _inputs()
    out = torch.zeros_like(q)
    lse = torch.zeros(2, 4, 5)
    with pytest.raises(ValueError, match="d_out"):
        ps.prefill_backward(q, k, v, out, lse, out[:, :4], qs, pl, 16)
    with pytest.raises(ValueError, match="lse"):
        ps.prefill_backward(q, k, v, out, lse.transpose(1, 2), out, qs, pl, 16)
    with pytest.raises(ValueError, match="out"):
        ps.prefill_backward(q, k, v, out[:1], lse, out, qs, pl, 16)


def test_consistent_shapes_reach_the_device_check(ps):
    # right shapes, CPU tensors: the next check (contiguous CUDA tensor) refuses
    q, k, v, qs, pl = _inputs()
    with pytest.raises(ValueError, match="CUDA"):
        ps.prefill(q, k, v, qs, pl, 16)


def test_ring_cache_slot_bases(ps):
    """Per-sequence pool bases: the pools end a capacity past the last base,
    rows_of follows the bases, and malformed bases are refused."""
    c = ps.RingCache(3, 2, 64, 8, [0, 0, 0], slot_base=[0, 5, 20], device="cpu")
    assert c.k_pool.shape[0] == 20 + c.capacity
    assert c.desc.total_slots == 20 + c.capacity
    assert c.slot_base.tolist() == [0, 5, 20]
    assert c.rows_of(1).tolist() == list(range(5, 5 + c.capacity))
    d = ps.RingCache(2, 2, 64, 8, [3, 1], device="cpu")  # default: s * capacity
    assert d.slot_base.tolist() == [0, d.capacity] and d.k_pool.shape[0] == 2 * d.capacity
    with pytest.raises(ValueError, match="slot_base"):
        ps.RingCache(3, 2, 64, 8, [0, 0, 0], slot_base=[0, 5], device="cpu")
    with pytest.raises(ValueError, match="slot_base"):
        ps.RingCache(2, 2, 64, 8, [0, 0], slot_base=[0, -1], device="cpu")
    with pytest.raises(ValueError, match="slot_base"):
        ps.RingCache(2, 2, 64, 8, [0, 0], slot_base=[0, 16], block_size=16, device="cpu")


def test_decode_graph_host_buffers_checked(ps):
    """DecodeGraph.step refuses host blocks of the wrong size, type or device
    before any call into the library."""
    with pytest.raises(ValueError, match="host_in"):
        ps.DecodeGraph._host(torch.zeros(10, dtype=torch.uint8), 11, "host_in")
    with pytest.raises(ValueError, match="host_res"):
        ps.DecodeGraph._host(torch.zeros(11, dtype=torch.int32), 11, "host_res")
    assert ps.DecodeGraph._host(None, 11, "host_in") is None
    assert ps.DecodeGraph._host(torch.zeros(11, dtype=torch.uint8), 11, "host_in").value
