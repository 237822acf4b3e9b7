"""The parity tolerance helpers against bf16 arithmetic done by torch (CPU)."""
import numpy as np
import torch

from _util import BF16_ARITH_SLACK, O_ABS, half_ulp_bf16, o_abs_bound


def _bf16_spacing(x: np.ndarray) -> np.ndarray:
    """Distance from each bf16 value to the next larger one, by bit increment."""
    b = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    nxt = (b.view(torch.int16) + 1).view(torch.bfloat16)
    return (nxt.double() - b.double()).numpy()


def test_half_ulp_matches_bf16_spacing():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(0.01, 60, 5000), 2.0 ** np.arange(-10, 6)])
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(half_ulp_bf16(xb), 0.5 * _bf16_spacing(xb))


def test_bound_is_one_hundredth_below_four():
    x = np.linspace(-3.98, 3.98, 2001)
    assert np.all(o_abs_bound(x) == O_ABS)


def test_bound_covers_bf16_rounding_of_large_outputs():
    """An exact value rounded to bf16 (what a perfect kernel returns) passes, with
    room for the arithmetic slack; the allowance is never larger than needed."""
    rng = np.random.default_rng(1)
    x = rng.uniform(3.9, 40, 20000) * rng.choice([-1, 1], 20000)
    xb = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    err = np.abs(xb - x)
    assert np.all(err + BF16_ARITH_SLACK <= o_abs_bound(x) + 1e-12)
    assert np.all(o_abs_bound(x) <= np.maximum(O_ABS, _bf16_spacing(np.abs(x) + O_ABS) / 2 * 1.0001
                                               + BF16_ARITH_SLACK))
