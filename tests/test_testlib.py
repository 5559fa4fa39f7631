"""CPU pins of the parity helpers the GPU tests rely on: the decision-boundary
band, the bf16 rounding-midpoint band and the outlier-list comparison (a
difference planted in the second argument must fail unless it sits in its
band)."""
import math

import numpy as np
import pytest

import tq_testlib as tl


def test_bf16_midpoint_band():
    # bf16 keeps 8 significant bits: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert tl.bf16_midpoint_band(1.0 + 2.0 ** -8)
    assert tl.bf16_midpoint_band(-(1.0 + 2.0 ** -8) * 2.0 ** -7)        # sign and scale free
    assert tl.bf16_midpoint_band((1.0 + 2.0 ** -8) * (1 + 5e-7))         # inside 1e-6
    assert not tl.bf16_midpoint_band((1.0 + 2.0 ** -8) * (1 + 3e-6))     # outside 1e-6
    assert not tl.bf16_midpoint_band(1.0)                                 # a bf16 value itself
    assert not tl.bf16_midpoint_band(1.0 + 2.0 ** -9)                     # a quarter step
    assert not tl.bf16_midpoint_band(0.0)
    # in [0.5, 1) the step is 2^-8: the midpoint above 0.75 is 0.75 + 2^-9
    assert tl.bf16_midpoint_band(0.75 + 2.0 ** -9)
    assert not tl.bf16_midpoint_band(0.75 + 2.0 ** -8)


def test_band_mask_uses_coordinate_scale_near_zero():
    d = 128
    t32 = np.array([-0.1, 0.0, 0.1], np.float32)
    y = np.array([0.1 * (1 + 5e-7), 0.1 * (1 + 5e-6), 0.5e-6 / math.sqrt(d), 5e-6 / math.sqrt(d)])
    np.testing.assert_array_equal(tl.band_mask(y, t32, d), [True, False, True, False])


def _enc(y, oval, is_out):
    return {"y": np.array([y], np.float64), "oval": np.array([oval], np.uint16),
            "is_out": np.array([is_out], np.uint8)}


def test_check_outliers_bands():
    d, T = 4, 2.0
    thr = T / math.sqrt(d)                      # 1.0
    mid = 1.0 + 2.0 ** -8                       # a bf16 midpoint above the threshold
    enc = _enc([mid, 3.0, thr * (1 + 1e-7), 0.2], [0x3F80, 0x4040, 0x3F80, 0], [1, 1, 1, 0])
    # identical lists: no band difference
    assert tl.check_outliers([{0: 0x3F80, 1: 0x4040, 2: 0x3F80}], enc, d, T) == 0
    # one bf16 step at the midpoint coordinate, and a threshold coordinate missing: two band differences
    assert tl.check_outliers([{0: 0x3F81, 1: 0x4040}], enc, d, T) == 2
    # one bf16 step where y is not at a midpoint: fails
    with pytest.raises(AssertionError):
        tl.check_outliers([{0: 0x3F80, 1: 0x4041, 2: 0x3F80}], enc, d, T)
    # two bf16 steps at the midpoint coordinate: fails
    with pytest.raises(AssertionError):
        tl.check_outliers([{0: 0x3F82, 1: 0x4040, 2: 0x3F80}], enc, d, T)
    # a coordinate far from the threshold missing: fails
    with pytest.raises(AssertionError):
        tl.check_outliers([{0: 0x3F80, 2: 0x3F80}], enc, d, T)
