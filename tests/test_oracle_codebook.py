"""Pins for the oracle's Gaussian Lloyd-Max codebook.

The oracle computes the table by Lloyd iteration with closed-form normal
integrals.  These tests check it against things that do not share its
arithmetic: the b = 1 closed form, Max's 1960 table, scipy quadrature of the
centroid condition and of the distortion, and the symmetry of the optimum.
"""
import math
import os

import numpy as np
import pytest
from scipy import integrate, stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "max1960_gaussian.txt")


def _max_table():
    tab = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        tab[(int(line[0]), line[1])] = [float(v) for v in line[2:]]
    return tab


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_matches_max_1960_table(orc, bits):
    K = 1 << bits
    c, t, mse, _ = orc.lloyd_max_gaussian(bits)
    tab = _max_table()
    # the table prints four significant figures
    np.testing.assert_allclose(c[K // 2:], tab[(K, "output")], rtol=6e-4, atol=0)
    if K > 2:
        np.testing.assert_allclose(t[K // 2:], tab[(K, "threshold")], rtol=6e-4, atol=0)
    assert mse == pytest.approx(tab[(K, "mse")][0], rel=1e-3)


def test_one_bit_closed_form(orc):
    c, t, mse, _ = orc.lloyd_max_gaussian(1)
    assert c[1] == pytest.approx(math.sqrt(2 / math.pi), abs=1e-13)
    assert c[0] == pytest.approx(-math.sqrt(2 / math.pi), abs=1e-13)
    assert t[0] == pytest.approx(0.0, abs=1e-15)
    assert mse == pytest.approx(1 - 2 / math.pi, abs=1e-13)


@pytest.mark.parametrize("bits,target", [(1, 0.3634), (2, 0.1175), (3, 0.03454), (4, 0.009497)])
def test_distortion_within_one_percent(orc, bits, target):
    _, _, mse, _ = orc.lloyd_max_gaussian(bits)
    assert abs(mse / target - 1) < 0.01


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_fixed_point_by_quadrature(orc, bits):
    """Each centroid is the conditional mean of its cell and each boundary the
    midpoint of its neighbours; the distortion equals the integral -- all by
    scipy quadrature, independent of the oracle's closed forms."""
    c, t, mse, _ = orc.lloyd_max_gaussian(bits)
    K = 1 << bits
    edges = [-np.inf] + list(t) + [np.inf]
    D = 0.0
    for k in range(K):
        a, b = edges[k], edges[k + 1]
        m0 = integrate.quad(stats.norm.pdf, a, b, epsabs=1e-14, epsrel=1e-13)[0]
        m1 = integrate.quad(lambda x: x * stats.norm.pdf(x), a, b, epsabs=1e-14, epsrel=1e-13)[0]
        assert m1 / m0 == pytest.approx(c[k], abs=1e-9)
        D += integrate.quad(lambda x: (x - c[k]) ** 2 * stats.norm.pdf(x), a, b,
                            epsabs=1e-14, epsrel=1e-13)[0]
    for k in range(K - 1):
        assert t[k] == pytest.approx(0.5 * (c[k] + c[k + 1]), abs=1e-15)
    assert D == pytest.approx(mse, rel=1e-8)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_symmetric_and_ascending(orc, bits):
    c, t, _, _ = orc.lloyd_max_gaussian(bits)
    np.testing.assert_allclose(c, -c[::-1], atol=1e-14)
    assert np.all(np.diff(c) > 0)
    # an odd number of boundaries; the middle one is exactly 0
    assert t[(1 << bits) // 2 - 1] == pytest.approx(0.0, abs=1e-15)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_f32_table_scaled_by_inverse_sqrt_d(orc, d, bits):
    """One unit-variance table per bit width scaled by 1/sqrt(d) (larql PR #196,
    turbo-quant note) -- not a sqrt(2)-narrow table."""
    c, _, _, _ = orc.lloyd_max_gaussian(bits)
    c32, t32 = orc.codebook_f32(bits, d)
    np.testing.assert_allclose(c32.astype(np.float64) * math.sqrt(d), c, rtol=1e-7)
    # boundaries: f32 midpoints of the f32 centroids
    mid = ((c32[:-1].astype(np.float64) + c32[1:].astype(np.float64)) / 2).astype(np.float32)
    np.testing.assert_array_equal(t32, mid)
    assert np.all(np.diff(c32) > 0) and np.all(c32[:-1] < t32) and np.all(t32 < c32[1:])
    # the sqrt(2)-narrow table the larql note fixed would put the outer 4-bit
    # centroid near 1.93/sqrt(d); ours sits at 2.733/sqrt(d)
    if bits == 4:
        assert c32[-1] * math.sqrt(d) == pytest.approx(2.733, abs=1e-3)
