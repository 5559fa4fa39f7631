"""Pins for the oracle's encode, record packing and decode."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _codec(orc, d=128, bits=3, T=0.0, cap=0):
    return orc.Codec(d=d, bits=bits, seed=1, T=T, cap=cap)


def _rows(n, d, seed=0, sigma=0.5):
    return synth.gaussian_bf16((n, d), seed, lognormal_sigma=sigma)


# --------------------------------------------------------------------------- encode


@pytest.mark.parametrize("d,bits", [(64, 1), (64, 3), (128, 2), (128, 3), (256, 4), (512, 4)])
def test_codes_are_nearest_centroid(orc, d, bits):
    """The midpoint comparison picks the nearest of the 2^b centroids (checked by
    brute-force argmin over squared distance), except at exact midpoint ties."""
    cod = _codec(orc, d, bits)
    enc = orc.encode_vectors(_rows(300, d, seed=d + bits), cod, want_y=True)
    c32, t32 = orc.codebook_f32(bits, d)
    y = enc["y"]
    dist = (y[..., None] - c32.astype(np.float64)[None, None, :]) ** 2
    nearest = np.argmin(dist, axis=-1)
    tie = np.min(np.abs(y[..., None] - t32.astype(np.float64)), axis=-1) < 1e-12
    assert np.array_equal(enc["codes"][~tie], nearest[~tie])


def test_rotation_is_unit_norm(orc):
    cod = _codec(orc, 128, 3)
    x = _rows(200, 128)
    enc = orc.encode_vectors(x, cod, want_y=True)
    np.testing.assert_allclose(np.linalg.norm(enc["y"], axis=1), 1.0, atol=1e-12)
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    np.testing.assert_array_equal(enc["norms"], np.linalg.norm(xd, axis=1).astype(np.float32))


def test_power_of_two_scaling_changes_only_the_norm(orc):
    cod = _codec(orc, 128, 3)
    x = _rows(256, 128)
    x2 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(4.0))  # exact in bf16
    a, b = orc.encode_vectors(x, cod), orc.encode_vectors(x2, cod)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(b["norms"], a["norms"] * np.float32(4.0))


def test_negation_mirrors_codes(orc):
    cod = _codec(orc, 128, 4)
    x = _rows(256, 128)
    xn = x ^ np.uint16(0x8000)
    a = orc.encode_vectors(x, cod, want_y=True)
    b = orc.encode_vectors(xn, cod)
    nz = a["y"] != 0.0
    np.testing.assert_array_equal(b["codes"][nz], 15 - a["codes"][nz])


@pytest.mark.parametrize("bits,D", [(2, 0.1175), (3, 0.03454), (4, 0.009497)])
def test_reconstruction_error_near_gaussian_distortion(orc, bits, D):
    """Relative squared error of decode(encode(x)) on the 4096x128 LogNormal
    workload sits near the Gaussian Lloyd-Max distortion D(b) (within 10%)."""
    cod = _codec(orc, 128, bits)
    x = synth.gaussian_bf16((4096, 128), 0, lognormal_sigma=0.5)
    rec = orc.encode_records(x, cod)
    xh = orc.decode_records(rec, 4096, cod)
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    rel = np.sum((xh - xd) ** 2, axis=1) / np.sum(xd ** 2, axis=1)
    assert abs(rel.mean() / D - 1) < 0.10


def test_zero_vector(orc):
    cod = _codec(orc, 128, 3, T=2.0)
    x = np.zeros((1, 128), np.uint16)
    enc = orc.encode_vectors(x, cod, want_y=True)
    assert enc["norms"][0] == 0.0
    assert np.all(enc["codes"] == 3) and not enc["is_out"].any()
    rec = orc.pack_records(enc, cod)
    assert np.all(orc.decode_records(rec, 1, cod) == 0.0)


@pytest.mark.parametrize("d", [64, 512])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_exact_ties_take_the_lower_code(orc, d, bits):
    """x = e_i + e_j with equal signs s_i = s_j: the rotated coordinate m is
    s_i (H_mi + H_mj) / sqrt(2 d), exactly 0 wherever H_mi != H_mj (half of
    them).  0 is the middle boundary of every table, and a value on a
    boundary takes the lower code: 2^(b-1) - 1.  Elsewhere |y| = sqrt(2/d)."""
    s = orc.signs(1, d)
    i, j = 0, next(k for k in range(1, d) if s[k] == s[0])
    x = np.zeros((1, d), np.uint16)
    x[0, i] = x[0, j] = 0x3F80                     # bf16 1.0
    enc = orc.encode_vectors(x, _codec(orc, d, bits), want_y=True)
    y = enc["y"][0]
    H = np.array([[(-1) ** bin(m & k).count("1") for k in (i, j)] for m in range(d)])
    zero = H[:, 0] != H[:, 1]
    assert zero.sum() == d // 2 and np.all(y[zero] == 0.0)
    np.testing.assert_allclose(np.abs(y[~zero]), np.sqrt(2.0 / d), rtol=1e-15)
    assert np.all(enc["codes"][0][zero] == (1 << (bits - 1)) - 1)
    t = orc.codebook_f32(bits, d)[1]
    assert t[(1 << (bits - 1)) - 1] == 0.0


def test_double_to_bf16_rounding(orc):
    """Round to nearest, ties to even, from the exact value (hand cases)."""
    one = 0x3F80
    assert orc.f64_to_bf16(1.0) == one
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8) == one                  # tie -> even (1.0)
    assert orc.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == one + 2          # tie -> even (1+2^-6)
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == one + 1  # above the tie
    assert orc.f64_to_bf16(-0.15625) == 0xBE20
    # a value whose f32 rounding would make a false tie: 1 + 2^-8 - 2^-30
    v = float(Fraction(1) + Fraction(1, 256) - Fraction(1, 2 ** 30))
    assert orc.f64_to_bf16(v) == one


# --------------------------------------------------------------------------- records


def test_bytes_per_vector(orc):
    c1 = _codec(orc, 128, 3)
    assert c1.record_bytes == 128 * 52                          # 48 B codes + 4 B norm
    gold = {l.split()[0]: int(l.split()[1]) for l in open(os.path.join(GOLD, "v4flash_bytes_per_token.txt"))
            if l.strip() and not l.startswith("#")}
    c3 = _codec(orc, 512, 4)
    assert c3.record_bytes / 128 == gold["turboquant_256_packed_f32_norm"]
    assert c3.record_bytes % 16 == 0 and c1.record_bytes % 16 == 0
    c4 = _codec(orc, 128, 4, T=2.0)
    lay = c4.layout()
    assert lay["norm"] == 128 * 64 and lay["count"] == lay["norm"] + 512
    assert lay["entries"] == lay["count"] + 128 and c4.outlier_cap == 1312
    assert c4.record_bytes == lay["entries"] + 4 * 1312


def test_packing_hand_example(orc):
    want = bytes.fromhex(" ".join(l for l in open(os.path.join(GOLD, "pack_d64_b3_ramp.txt"))
                                  if not l.startswith("#")))
    cod = _codec(orc, 64, 3)
    enc = dict(codes=np.tile(np.arange(8, dtype=np.uint8), 8)[None, :],
               norms=np.ones(1, np.float32), is_out=np.zeros((1, 64), np.uint8),
               oval=np.zeros((1, 64), np.uint16))
    rec = orc.pack_records(enc, cod)
    assert bytes(rec[0, :24]) == want
    assert [orc.read_code(rec[0, :24], j, 3) for j in range(64)] == list(range(8)) * 8
    np.testing.assert_array_equal(rec[0, 128 * 24:128 * 24 + 4].view(np.float32), [1.0])


def test_constant_code_decodes_to_first_axis(orc):
    """All codes k, norm n: yhat = c_k * ones, H(ones)/sqrt(d) = sqrt(d) e_0, so
    xhat = n * c_k * sqrt(d) * s_0 * e_0 (closed form)."""
    d, bits, k, n = 128, 4, 13, 3.5
    cod = _codec(orc, d, bits)
    enc = dict(codes=np.full((1, d), k, np.uint8), norms=np.array([n], np.float32),
               is_out=np.zeros((1, d), np.uint8), oval=np.zeros((1, d), np.uint16))
    rec = orc.pack_records(enc, cod)
    c32, _ = orc.codebook_f32(bits, d)
    s = orc.signs(1, d)
    xh = orc.decode_records(rec, 1, cod)[0]
    want = np.zeros(d); want[0] = n * float(c32[k]) * math.sqrt(d) * s[0]
    np.testing.assert_allclose(xh, want, atol=1e-12)
    np.testing.assert_allclose(orc.decode_records(rec, 1, cod, rotated=True)[0],
                               n * np.full(d, float(c32[k])), atol=0)


def test_decode_inverts_the_rotation(orc):
    """decode = n * s . H(yhat)/sqrt(d): re-rotating the decoded vector gives back
    n * yhat exactly up to fp64 rounding."""
    cod = _codec(orc, 256, 3, T=2.0)
    x = _rows(130, 256, seed=3)
    rec = orc.encode_records(x, cod)
    xh = orc.decode_records(rec, 130, cod)
    yr = orc.decode_records(rec, 130, cod, rotated=True)
    s = orc.signs(1, 256).astype(np.float64)
    np.testing.assert_allclose(orc.fwht(s * xh), yr, atol=1e-11)


# --------------------------------------------------------------------------- outliers


def test_outlier_set_and_values(orc):
    d = 128
    cod = _codec(orc, d, 4, T=2.0)
    x = synth.gaussian_bf16((256, d), 5, outlier_frac=0.02)
    enc = orc.encode_vectors(x, cod, want_y=True)
    y = enc["y"]
    np.testing.assert_array_equal(enc["is_out"].astype(bool), np.abs(y) > 2.0 / math.sqrt(d))
    # about 4.55% of N(0,1) coordinates exceed 2 sigma
    assert 0.03 < enc["is_out"].mean() < 0.06
    for i, j in zip(*np.nonzero(enc["is_out"][:20])):
        assert enc["oval"][i, j] == orc.f64_to_bf16(y[i, j])
    rec = orc.pack_records(enc, cod)
    lay = cod.layout()
    counts = rec[:, lay["count"]:lay["count"] + 128].reshape(-1)[:256]
    np.testing.assert_array_equal(counts, enc["is_out"].sum(axis=1))
    # decode replaces the centroid by the stored value before the inverse WHT
    yr = orc.decode_records(rec, 256, cod, rotated=True)
    norms = enc["norms"].astype(np.float64)[:, None]
    oi = enc["is_out"].astype(bool)
    np.testing.assert_allclose(yr[oi], (norms * orc.bf16_to_f64(enc["oval"]))[oi], rtol=1e-15)


def test_infinite_threshold_is_the_plain_codec(orc):
    x = _rows(200, 128, seed=9)
    plain, inf = _codec(orc, 128, 3), _codec(orc, 128, 3, T=float("inf"))
    rp, ri = orc.encode_records(x, plain), orc.encode_records(x, inf)
    n_code = 128 * 48 + 512
    np.testing.assert_array_equal(rp[:, :n_code], ri[:, :n_code])
    assert not ri[:, n_code:n_code + 128].any()
    np.testing.assert_array_equal(orc.decode_records(rp, 200, plain), orc.decode_records(ri, 200, inf))


def test_outlier_capacity_overflow(orc):
    """Entries fill in (slot, index) order up to the record capacity; the rest
    keep their ordinary codes."""
    d, cap = 64, 8
    cod = _codec(orc, d, 2, T=0.5, cap=cap)
    x = _rows(5, d, seed=11)
    enc = orc.encode_vectors(x, cod, want_y=True)
    rec = orc.pack_records(enc, cod)
    lay = cod.layout()
    counts = rec[0, lay["count"]:lay["count"] + 5].astype(int)
    raw = enc["is_out"].sum(axis=1)
    assert raw.sum() > cap and counts.sum() == cap
    want, left = [], cap
    for r in raw:
        want.append(min(r, left)); left -= want[-1]
    assert list(counts) == want
    ent = rec[0, lay["entries"]:lay["entries"] + 4 * cap].reshape(cap, 4)
    idx = ent[:, 0].astype(int) | (ent[:, 1].astype(int) << 8)
    exp = [j for i in range(5) for j in np.nonzero(enc["is_out"][i])[0]][:cap]
    assert list(idx) == exp
