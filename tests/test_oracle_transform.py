"""Pins for the oracle's sign diagonal and orthonormal Walsh-Hadamard transform."""
import os

import numpy as np
import pytest
from scipy.linalg import hadamard

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed0.txt")


def test_splitmix64_published_vectors(orc):
    want = [int(l, 16) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    got = [int(v) for v in orc.splitmix64(0, len(want))]
    assert got == want


def test_signs_are_top_bits_and_prefix_stable(orc):
    outs = orc.splitmix64(1, 512)
    s = orc.signs(1, 512)
    np.testing.assert_array_equal(s, np.where((outs >> np.uint64(63)) == 1, -1, 1))
    # the sign vector of a smaller head dim is a prefix of the larger one
    np.testing.assert_array_equal(orc.signs(1, 64), s[:64])
    assert set(np.unique(s)) == {-1, 1}
    assert not np.array_equal(orc.signs(2, 128), orc.signs(1, 128))


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_equals_sylvester_matrix(orc, d):
    """Natural (Sylvester) order, orthonormal: scipy's hadamard(d)/sqrt(d)."""
    x = np.random.default_rng(d).standard_normal((3, d))
    H = hadamard(d).astype(np.float64) / np.sqrt(d)
    np.testing.assert_allclose(orc.fwht(x), x @ H.T, atol=1e-12)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_involution_parseval_and_basis(orc, d):
    rng = np.random.default_rng(7 + d)
    x32 = rng.standard_normal((16, d)).astype(np.float32)
    x = x32.astype(np.float64)
    y = orc.fwht(x)
    # Parseval
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # randomized Hadamard round trip without quantization: s . H(H(s . x)) = x
    s = orc.signs(1, d).astype(np.float64)
    back = s * orc.fwht(orc.fwht(s * x))
    assert np.max(np.abs(back - x)) < 1e-6 * max(1.0, np.max(np.abs(x)))
    assert np.max(np.abs(back - x)) < 1e-12
    # H e_0 = 1/sqrt(d) * ones;  H ones = sqrt(d) e_0
    e0 = np.zeros(d); e0[0] = 1
    np.testing.assert_allclose(orc.fwht(e0), np.full(d, 1 / np.sqrt(d)), atol=1e-15)
    np.testing.assert_allclose(orc.fwht(np.ones(d)), np.sqrt(d) * e0, atol=1e-12)
