"""CPU oracle for Prefix-Sliding attention (float64, slow, plain).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the library.  It shares
no code with the CUDA path.

Pinned functions (each checked in ``tests/test_oracle_pins.py`` against
something other than itself):
  round_bf16        torch's float32 -> bfloat16 cast; hand-made ties
  rope              norm preservation, relative-position invariance, a hand
                    computed D=4 case, identity at position 0
  allowed / visible_positions
                    key count = min(p+1, P+W) by brute force; the pages' cap of
                    4,196 keys for a 100-token prefix and a 4,096 window
  masked_attention  torch scaled_dot_product_attention (causal and banded)
                    in float64; one-key and uniform-key closed forms
  attend            W >= length reduces to causal attention, P = 0 to a plain
                    sliding window; pure-Python enumeration on tiny inputs
  ring_slot / RingSim
                    live set equals the mask's visible set after every append
                    (thousands of evictions), slot range [0, P+W)
  tile_classes      sum of admitted pairs equals the closed-form total; the
                    pages' skip rule (no admitted element) checked per tile
  reset_positions / attend_reset_pe
                    pure-Python enumeration that rotates every key at its
                    renumbered position; equals attend while nothing has been
                    evicted; window-only keys (P = 0) are a uniform shift
  attend_backward   torch autograd of scaled_dot_product_attention in float64
                    (explicit mask, GQA by repeat), also for chunks at offset
                    positions; central finite differences of the forward through
                    RoPE; its forward equals attend
  attend_backward_at
                    torch autograd of scaled_dot_product_attention (selected
                    rows of dq, dk, dv), at position 0 and at an offset
"""
from .prefix_sliding import (  # noqa: F401
    FULL, PARTIAL, SKIP, RingSim, allowed, attend, attend_backward, attend_backward_at,
    attend_reset_pe, masked_attention,
    reset_positions, ring_slot, rope, round_bf16, tile_classes, visible_positions,
)
