"""Pins of the oracle's per-vector scale variants and caller-supplied centroid
tables.  Sources: the turboquant_plus commit log (the EDEN-scale commits: the
inner-product-preserving scale ||x||^2/<c,x>, the least-squares scale
<c,x>/||c||^2, and the Appendix A note that their geometric mean is the
matched-norm scale ||x||/||c||); "v1.3 PPL on vLLM" (PR #15), the calibrated
Lloyd-Max commit (a caller-supplied sorted 2^b f32 table replacing the
Gaussian one).  Each scale is pinned by the property that defines it, checked
on the oracle's own decode, not by re-typing its formula."""
import math

import numpy as np
import pytest

import synth

MODES = ("matched_norm", "inner_product", "least_squares")


def _rows(n, d, seed, **kw):
    return synth.gaussian_bf16((n, d), seed, lognormal_sigma=0.5, **kw)


def _decode(orc, x, cod):
    rec = orc.encode_records(x, cod)
    return orc.decode_records(rec, x.shape[0], cod)


@pytest.mark.parametrize("d,bits,T", [(64, 2, 0.0), (128, 3, 0.0), (128, 4, 2.0), (512, 4, 0.0)])
def test_scale_modes_keep_codes_and_outliers(orc, d, bits, T):
    x = _rows(200, d, 5 + d + bits, outlier_frac=0.02 if T else 0.0)
    base = orc.encode_vectors(x, orc.Codec(d=d, bits=bits, T=T))
    for m in MODES:
        e = orc.encode_vectors(x, orc.Codec(d=d, bits=bits, T=T, scale=m))
        for k in ("codes", "is_out", "oval"):
            np.testing.assert_array_equal(e[k], base[k])


@pytest.mark.parametrize("d,bits,T", [(64, 2, 0.0), (128, 3, 0.0), (128, 4, 2.0), (512, 1, 0.0)])
def test_scale_modes_defining_properties(orc, d, bits, T):
    """matched norm: ||xhat|| = ||x||; inner product: <xhat, x> = ||x||^2;
    least squares: the residual x - xhat is orthogonal to xhat (the normal
    equation of min_S ||x - S c||^2), and its error is the smallest of all
    four scales for every vector."""
    x = _rows(200, d, 11 + d + bits, outlier_frac=0.02 if T else 0.0)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    nx = np.linalg.norm(xf, axis=1)
    dec = {m: _decode(orc, x, orc.Codec(d=d, bits=bits, T=T, scale=m)) for m in ("norm",) + MODES}
    # the stored scale is f32: relative agreement to a few f32 roundings
    np.testing.assert_allclose(np.linalg.norm(dec["matched_norm"], axis=1), nx, rtol=2e-7)
    np.testing.assert_allclose(np.sum(dec["inner_product"] * xf, axis=1), nx ** 2, rtol=2e-7)
    ls = dec["least_squares"]
    assert np.max(np.abs(np.sum((xf - ls) * ls, axis=1)) / nx ** 2) < 1e-6
    err = {m: np.sum((xf - v) ** 2, axis=1) for m, v in dec.items()}
    for m in ("norm", "matched_norm", "inner_product"):
        assert np.all(err["least_squares"] <= err[m] * (1 + 1e-6) + 1e-12), m


def test_geometric_mean_identity(orc):
    """sqrt(S_inner_product * S_least_squares) = S_matched_norm (Appendix A note)."""
    d, bits = 128, 3
    x = _rows(300, d, 21)
    S = {m: orc.encode_vectors(x, orc.Codec(d=d, bits=bits, scale=m))["norms"].astype(np.float64) for m in MODES}
    np.testing.assert_allclose(np.sqrt(S["inner_product"] * S["least_squares"]), S["matched_norm"], rtol=3e-7)


def test_scales_agree_when_the_quantised_vector_is_parallel(orc):
    """x = 3 e_0 rotates to y = +-1/sqrt(d) in every coordinate; at one bit each
    coordinate dequantises to +-sqrt(2/pi)/sqrt(d) with y's sign, so chat is
    parallel to y and all four scales are n / sqrt(2/pi) except the plain one,
    which stays n = 3."""
    d = 64
    x = np.zeros((1, d), np.uint16)
    x[0, 0] = synth.f32_to_bf16_bits(np.array([3.0], np.float32))[0]
    want = 3.0 / math.sqrt(2.0 / math.pi)
    for m in MODES:
        S = float(orc.encode_vectors(x, orc.Codec(d=d, bits=1, scale=m))["norms"][0])
        assert S == pytest.approx(want, rel=2e-7), m
    assert float(orc.encode_vectors(x, orc.Codec(d=d, bits=1))["norms"][0]) == 3.0


def test_zero_vector_scale_is_zero(orc):
    x = np.zeros((2, 128), np.uint16)
    for m in MODES:
        e = orc.encode_vectors(x, orc.Codec(d=128, bits=3, scale=m))
        assert np.all(e["norms"] == 0.0)


def _table(bits, d):
    """A symmetric ascending table that is not the Gaussian one (wider outer levels)."""
    half = np.linspace(0.15, 2.2, 1 << (bits - 1)) ** 1.2
    return tuple(float(v) for v in np.float32(np.concatenate([-half[::-1], half]) / math.sqrt(d)))


def test_custom_table_equal_to_gaussian_is_the_default(orc):
    d, bits = 128, 3
    c, _ = orc.codebook_f32(bits, d)
    x = _rows(300, d, 31)
    a = orc.encode_records(x, orc.Codec(d=d, bits=bits))
    b = orc.encode_records(x, orc.Codec(d=d, bits=bits, centroids=tuple(float(v) for v in c)))
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("d,bits", [(64, 2), (128, 3), (256, 4)])
def test_custom_table_codes_are_nearest_centroid(orc, d, bits):
    """With a caller's table the codes are the nearest of its centroids (brute
    force over the table on the exact rotated values), and decode dequantises
    through that table."""
    tab = _table(bits, d)
    cod = orc.Codec(d=d, bits=bits, centroids=tab)
    x = _rows(300, d, 41 + d)
    enc = orc.encode_vectors(x, cod, want_y=True)
    c = np.array(tab, np.float64)
    near = np.argmin(np.abs(enc["y"][..., None] - c), axis=-1)
    t = orc.midpoints_f32(bits, np.array(tab, np.float32)).astype(np.float64)
    tie = np.any(np.abs(enc["y"][..., None] - t) < 1e-12, axis=-1)
    assert np.all((enc["codes"] == near) | tie)
    rec = orc.pack_records(enc, cod)
    rot = orc.decode_records(rec, 300, cod, rotated=True)
    np.testing.assert_allclose(rot, enc["norms"][:, None].astype(np.float64) * c[enc["codes"]], rtol=0, atol=0)
