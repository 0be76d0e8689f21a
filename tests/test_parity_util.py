"""Pins of the parity gate's bf16 rounding measure (CPU).

`bf16_rounding_excess(o, o_ref)` is the distance from o_ref to the interval of
reals that round to the bf16 value o. Pinned here against an independent
construction of that interval from the bit patterns of o's two bf16
neighbours, and against torch's own rounding: the excess is 0 exactly when
o_ref (a float32 value, so that one rounding step is involved) rounds to o.
"""
import numpy as np
import torch

from parity_util import bf16_rounding_excess


def _neighbours(y_bf16: torch.Tensor):
    """The bf16 values just below and just above each (finite, nonzero) y,
    from the 16-bit patterns: magnitude +-1 in the integer encoding."""
    bits = y_bf16.view(torch.int16).to(torch.int32)
    mag = bits & 0x7FFF
    sign = bits & 0x8000
    up_mag, down_mag = mag + 1, mag - 1   # next larger / smaller magnitude

    def from_bits(m):
        return (sign | m).to(torch.int16).view(torch.bfloat16).double()

    pos = y_bf16.double() > 0
    above = torch.where(pos, from_bits(up_mag), from_bits(down_mag))
    below = torch.where(pos, from_bits(down_mag), from_bits(up_mag))
    return below, above


def test_excess_equals_distance_to_the_rounding_interval():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(4000) * 4, rng.standard_normal(1000) * 1e-3,
                           [1.0, 2.0, 4.0, -2.0, 0.5, -0.25, 3.984375, -4.0, 8.0, 1.0078125]])
    y = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    y = y[y != 0]
    below, above = _neighbours(y)
    yd = y.double()
    lo, hi = ((below + yd) / 2).numpy(), ((yd + above) / 2).numpy()
    for spread in (1e-4, 3e-3, 1e-2, 5e-2):
        r = yd.numpy() + rng.uniform(-1, 1, yd.shape) * spread * np.maximum(1.0, np.abs(yd.numpy()))
        expect = np.maximum(0.0, np.maximum(lo - r, r - hi))
        got = bf16_rounding_excess(yd.numpy(), r)
        np.testing.assert_allclose(got, expect, rtol=1e-12, atol=1e-300)


def test_excess_is_zero_exactly_when_the_reference_rounds_to_the_value():
    rng = np.random.default_rng(1)
    r32 = (rng.standard_normal(20000) * 4).astype(np.float32)
    # a random bf16 value near each reference: its own rounding or a neighbour
    rn = torch.from_numpy(r32).to(torch.bfloat16)
    below, above = _neighbours(rn)
    pick = rng.integers(0, 3, r32.shape)
    cand = torch.where(torch.from_numpy(pick == 0), below, torch.where(torch.from_numpy(pick == 1), rn.double(), above))
    ex = bf16_rounding_excess(cand.numpy(), r32.astype(np.float64))
    rounds_to = cand.numpy() == rn.double().numpy()
    assert np.all((ex == 0) == rounds_to)
    # the stored value's own rounding interval is at most half a neighbour gap away
    assert np.all(ex[~rounds_to] <= (above - below).abs().numpy()[~rounds_to])


def test_excess_of_zero_is_the_magnitude():
    assert bf16_rounding_excess(np.array([0.0, 0.0]), np.array([0.003, -0.02])).tolist() == [0.003, 0.02]
