"""GPU parity of the codebook, encode and decode kernels against the oracle,
called through the C ABI (Python binding)."""
import math

import numpy as np
import pytest

import synth
import tq_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rotated_lloyd_max_gb300 import build
    build.build()
    import rotated_lloyd_max_gb300 as m
    m.load()
    return m


def _ocodec(orc, c):
    return orc.Codec(d=c.head_dim, bits=c.bits, seed=int(c.c.sign_seed), T=float(c.c.outlier_T),
                     cap=int(c.c.outlier_cap) if c.c.outlier_T else 0)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(tq, orc, d, bits):
    c = tq.tq_make_codebook(bits, d, sign_seed=1)
    c32, t32 = orc.codebook_f32(bits, d)
    np.testing.assert_array_equal(np.array(c.centroids(), np.float32), c32)
    np.testing.assert_array_equal(np.array(c.boundaries(), np.float32), t32)
    s = orc.signs(1, d)
    words = np.array(c.sign_words(), np.uint32)
    got = np.array([-1 if (words[j // 32] >> (j % 32)) & 1 else 1 for j in range(d)], np.int8)
    np.testing.assert_array_equal(got, s)
    assert c.mse == pytest.approx(orc.lloyd_max_gaussian(bits)[2], rel=1e-12)
    assert c.record_bytes == orc.Codec(d=d, bits=bits).record_bytes


DECODE_TOL = 1e-5   # max-abs, decoded f32 against the oracle's fp64 decode of the same records


def _check_decode(got, want, what):
    """Decoded vectors within 1e-5 max-abs of the oracle.  Vectors that miss
    are listed with their scale n * max|yhat| (= max|xhat| up to the
    transform) before the assertion fails; the relative error is printed as
    a second figure."""
    err = np.abs(got.astype(np.float64) - want).max(axis=1)
    scale = np.abs(want).max(axis=1)
    rel = float((err / np.maximum(scale, 1e-30)).max())
    print(f"decode {what}: max-abs {err.max():.3e}, max relative {rel:.3e}, max |xhat| {scale.max():.2f}")
    bad = np.nonzero(err > DECODE_TOL)[0]
    for i in bad[:20]:
        print(f"  vector {i}: max-abs {err[i]:.3e}, max |xhat| {scale[i]:.2f}")
    assert bad.size == 0, f"{bad.size} decoded vectors beyond {DECODE_TOL} max-abs"


def _encode_gpu(tq, c, x_bits, groups=1, first_vec=0, canary=0xAB):
    import torch
    n = x_bits.shape[-2]
    nrec = (first_vec + n + 127) // 128
    src = tl.to_bf16_tensor(x_bits, "cuda")
    dst = torch.full((groups, nrec + 1, c.record_bytes), canary, dtype=torch.uint8, device="cuda")
    tq.tq_encode(c, src.reshape(groups, n, c.head_dim), dst, first_vec=first_vec)
    torch.cuda.synchronize()
    return dst.cpu().numpy()


def test_codec_roundtrip_workload(tq, orc):
    """4096 x 128 bf16, N(0,1) x LogNormal(0, 0.5), b = 3: codes match the
    oracle outside the boundary band, norms within 2 ulp, 52 B/vector, and the
    reconstruction error sits at the Gaussian Lloyd-Max distortion."""
    import torch
    c = tq.tq_make_codebook(3, 128, sign_seed=1)
    oc = _ocodec(orc, c)
    x = synth.gaussian_bf16((4096, 128), 0, lognormal_sigma=0.5)
    rec = _encode_gpu(tq, c, x)[0]
    assert c.record_bytes == 128 * 52
    codes, norms, _ = tl.unpack_records(rec, 4096, 128, 3)
    enc = orc.encode_vectors(x, oc, want_y=True)
    mism, band = tl.check_codes(codes, enc, orc.codebook_f32(3, 128)[1], 128)
    tl.check_norms(norms, enc)
    # records beyond the written ones are untouched
    assert np.all(rec[32:] == 0xAB)
    # decode on the GPU and compare with the oracle decode of the same records
    out = torch.empty((4096, 128), dtype=torch.float32, device="cuda")
    tq.tq_decode(c, torch.from_numpy(rec).cuda(), out)
    got = out.cpu().numpy()
    want = orc.decode_records(rec, 4096, oc)
    _check_decode(got, want, "codec round trip")
    xd = synth.bf16_bits_to_f32(x).astype(np.float64)
    rel = (np.sum((got - xd) ** 2, 1) / np.sum(xd ** 2, 1)).mean()
    assert abs(rel / 0.03454 - 1) < 0.10


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("mode", ["plain", "offset", "outliers"])
def test_encode_decode_parity(tq, orc, d, bits, mode):
    """Ragged sizes spanning several records, two groups, an unaligned start
    (no outliers) or an outlier side list (T = 2 on data with 2% N(0,36)
    coordinates); decode cross-paired on the GPU's records."""
    import torch
    T = 2.0 if mode == "outliers" else 0.0
    first = 37 if mode == "offset" else 0
    n, groups = 300, 2
    c = tq.tq_make_codebook(bits, d, sign_seed=1, outlier_T=T)
    oc = _ocodec(orc, c)
    x = synth.gaussian_bf16((groups, n, d), 1000 + d + bits, outlier_frac=0.02 if T else 0.0,
                            lognormal_sigma=0.5)
    rec = _encode_gpu(tq, c, x, groups=groups, first_vec=first)
    t32 = orc.codebook_f32(bits, d)[1]
    for g in range(groups):
        # the oracle packs tokens 0..first+n-1; compare the written tokens
        codes, norms, outs = tl.unpack_records(rec[g], first + n, d, bits, T != 0.0, oc.outlier_cap if T else 0)
        enc = orc.encode_vectors(x[g], oc, want_y=True)
        tl.check_norms(norms[first:], enc)
        band = tl.check_codes(codes[first:], enc, t32, d, total_frac=None)[0]
        if T:
            band += tl.check_outliers(outs, enc, d, T)
        assert band <= max(1, 1e-5 * n * d), f"{band} band differences"
        # slots before `first` in the first record and records past the end keep the canary
        if first:
            rb = d * bits // 8
            assert np.all(rec[g, 0, :first * rb] == 0xAB)
        assert np.all(rec[g, (first + n + 127) // 128:] == 0xAB)
        dst = torch.empty((n, d), dtype=torch.float32, device="cuda")
        tq.tq_decode(c, torch.from_numpy(np.ascontiguousarray(rec[g])).cuda(), dst, first_vec=first)
        got = dst.cpu().numpy()
        # oracle decode of the GPU's own records (cross-pairing isolates decode numerics)
        full = orc.decode_records(rec[g], first + n, oc)[first:]
        _check_decode(got, full, f"d {d} b {bits} {mode} group {g}")


@pytest.mark.parametrize("n_rec,first,T", [(3, 37, 0.0), (3, 0, 2.0), (40, 0, 2.0), (200, 5, 0.0), (200, 0, 2.0)])
def test_decode_record_splits(tq, orc, n_rec, first, T):
    """Decodes of fewer records than SMs split each record over 4 CTAs of 32
    slots (3 and 40 records); 200 records keep one CTA each. Every slot,
    including a ragged start and end, decodes as the oracle does from the
    same records (outlier codecs start at a record boundary)."""
    import torch
    d, bits = 128, 3
    c = tq.tq_make_codebook(bits, d, sign_seed=1, outlier_T=T)
    oc = _ocodec(orc, c)
    n = n_rec * 128 - first - 11                      # a ragged end in the last record
    x = synth.gaussian_bf16((1, n, d), 77 + n_rec, outlier_frac=0.02 if T else 0.0, lognormal_sigma=0.5)
    rec = _encode_gpu(tq, c, x, first_vec=first)[0]
    dst = torch.empty((n, d), dtype=torch.float32, device="cuda")
    tq.tq_decode(c, torch.from_numpy(np.ascontiguousarray(rec)).cuda(), dst, first_vec=first)
    got = dst.cpu().numpy()
    want = orc.decode_records(rec, first + n, oc)[first:]
    _check_decode(got, want, f"{n_rec} records from slot {first}")


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_zero_vectors(tq, orc, d):
    """Zero vectors beside a nonzero one in the same tile: code of 0, norm 0,
    no side-list entries, decoded to exact zeros; the nonzero vector as the oracle."""
    import torch
    c = tq.tq_make_codebook(3, d, sign_seed=1, outlier_T=2.0)
    x = np.zeros((130, d), np.uint16)
    x[5] = synth.gaussian_bf16((1, d), 3)[0]
    rec = _encode_gpu(tq, c, x)[0]
    codes, norms, outs = tl.unpack_records(rec, 130, d, 3, True, c.c.outlier_cap)
    zero = np.ones(130, bool); zero[5] = False
    assert np.all(codes[zero] == 3) and np.all(norms[zero] == 0) and all(not outs[i] for i in np.nonzero(zero)[0])
    enc = orc.encode_vectors(x[5:6], _ocodec(orc, c), want_y=True)
    tl.check_norms(norms[5:6], enc)
    tl.check_codes(codes[5:6], enc, orc.codebook_f32(3, d)[1], d, total_frac=None)
    assert tl.check_outliers([outs[5]], enc, d, 2.0) <= 1
    dst = torch.empty((130, d), dtype=torch.float32, device="cuda")
    tq.tq_decode(c, torch.from_numpy(rec).cuda(), dst)
    assert torch.all(dst[torch.from_numpy(zero).cuda()] == 0)


def test_sweep_sample_parity(tq, orc):
    """Encode sweep shapes (d x b) on 2^16 N(0,1) vectors: all codes and norms
    against the oracle."""
    import torch
    n = 1 << 16
    for d in (64, 128, 256, 512):
        x = synth.gaussian_bf16((n, d), 7 + d)
        for bits in (2, 3, 4):
            c = tq.tq_make_codebook(bits, d, sign_seed=1)
            rec = _encode_gpu(tq, c, x)[0]
            codes, norms, _ = tl.unpack_records(rec, n, d, bits)
            enc = orc.encode_vectors(x, _ocodec(orc, c), want_y=True)
            tl.check_codes(codes, enc, orc.codebook_f32(bits, d)[1], d)
            tl.check_norms(norms, enc)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("mode", ["matched_norm", "inner_product", "least_squares"])
@pytest.mark.parametrize("T", [0.0, 2.0])
def test_scale_modes(tq, orc, d, mode, T):
    """The per-vector scale variants (turboquant_plus commit log, the EDEN-scale
    commits): codes and outlier lists as in the plain codec, the stored f32
    scale within 4e-6 relative of the oracle's (f32 sums of at most 512
    positive terms against fp64) on every vector whose codes match, and the
    GPU decode of those records within 1e-5 of the oracle's."""
    import torch
    bits = 3
    c = tq.with_scale(tq.tq_make_codebook(bits, d, sign_seed=1, outlier_T=T), mode)
    oc = orc.Codec(d=d, bits=bits, seed=1, T=T, cap=int(c.c.outlier_cap) if T else 0, scale=mode)
    n = 300
    x = synth.gaussian_bf16((n, d), 2000 + d, outlier_frac=0.02 if T else 0.0, lognormal_sigma=0.5)
    rec = _encode_gpu(tq, c, x)[0]
    codes, norms, outs = tl.unpack_records(rec, n, d, bits, T != 0.0, oc.outlier_cap if T else 0)
    enc = orc.encode_vectors(x, oc, want_y=True)
    band = tl.check_codes(codes, enc, orc.codebook_f32(bits, d)[1], d, total_frac=None)[0]
    if T:
        band += tl.check_outliers(outs, enc, d, T)
    assert band <= max(1, 1e-5 * n * d)
    same = np.all(codes == enc["codes"], axis=1)
    if T:
        same &= np.array([set(o) == set(np.nonzero(enc["is_out"][i])[0]) for i, o in enumerate(outs)])
    assert same.sum() >= n - 2
    np.testing.assert_allclose(norms[same], enc["norms"][same], rtol=4e-6)
    dst = torch.empty((n, d), dtype=torch.float32, device="cuda")
    tq.tq_decode(c, torch.from_numpy(rec).cuda(), dst)
    _check_decode(dst.cpu().numpy(), orc.decode_records(rec, n, oc), f"d {d} {mode} T {T}")
