"""The seeded input generators follow the stated recipes: N(0,1) rows,
per-row LogNormal(0, sigma) scales, a few fixed channels per group scaled x 8,
a fraction of coordinates from N(0, 36), bf16 round-to-nearest-even; both the
host (numpy) and the device-side (torch) generator, the latter run on the CPU
here.  Statistical checks with wide margins, fixed seeds."""
import numpy as np
import pytest
import torch

import synth


def _f32(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _torch(shape, seed, **kw):
    t = synth.torch_gaussian_bf16(shape, seed, "cpu", **kw)
    return t.to(torch.float32).numpy().astype(np.float64)


@pytest.fixture(params=["numpy", "torch"])
def draw(request):
    if request.param == "numpy":
        return lambda shape, seed, **kw: _f32(synth.gaussian_bf16(shape, seed, **kw))
    return _torch


def test_standard_normal(draw):
    x = draw((4096, 128), 0)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    assert abs(np.mean(np.abs(x) > 2) - 0.0455) < 0.003      # two-sided 2-sigma tail of N(0,1)


def test_per_row_lognormal_scale(draw):
    """Rows of N(0,1) x LogNormal(0, 0.5): log of the row rms is N(0, 0.5^2)."""
    x = draw((8192, 128), 1, lognormal_sigma=0.5)
    lr = np.log(np.sqrt(np.mean(x ** 2, axis=1)))
    assert abs(lr.std() - 0.5) < 0.03 and abs(lr.mean()) < 0.03


def test_fixed_channels(draw):
    """4 channels per (layer, head) group scaled x 8, the same channels for every
    row of the group, different groups drawing their own."""
    x = draw((3, 2, 2048, 128), 2, fixed_channels=4)
    sets = []
    for g in np.ndindex(3, 2):
        rms = np.sqrt(np.mean(x[g] ** 2, axis=0))
        hot = np.flatnonzero(rms > 4)
        assert len(hot) == 4
        assert np.all(np.abs(rms[hot] - 8) < 1) and np.all(np.abs(np.delete(rms, hot) - 1) < 0.15)
        sets.append(tuple(hot))
    assert len(set(sets)) > 1


def test_outlier_fraction(draw):
    """2% of coordinates from N(0, 36): the fraction beyond 4 is about
    0.02 * P(|N(0,36)| > 4) + 0.98 * P(|N(0,1)| > 4) = 0.0101."""
    x = draw((4096, 128), 3, outlier_frac=0.02)
    frac = np.mean(np.abs(x) > 4)
    assert abs(frac - 0.0101) < 0.0015


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5], np.float32)
    got = synth.f32_to_bf16_bits(vals)
    # the bf16 spacing at 1 is 2^-7: 1 + 2^-8 is a tie between 0x3F80 and 0x3F81 and goes
    # to the even 0x3F80; 1 + 3 * 2^-8 ties between 0x3F81 and 0x3F82 and goes to 0x3F82
    assert list(got[:4]) == [0x3F80, 0x3F80, 0x3F82, 0x3F80]
    assert got[4] == 0xC020
    assert np.array_equal(synth.bf16_bits_to_f32(got[:5]), np.float32([1.0, 1.0, 1.015625, 1.0, -2.5]))


def test_same_seed_same_draw():
    a = synth.gaussian_bf16((64, 64), 7, lognormal_sigma=0.3, fixed_channels=2)
    b = synth.gaussian_bf16((64, 64), 7, lognormal_sigma=0.3, fixed_channels=2)
    assert np.array_equal(a, b)
    c = synth.torch_gaussian_bf16((64, 64), 7, "cpu")
    d = synth.torch_gaussian_bf16((64, 64), 7, "cpu")
    assert torch.equal(c, d)


def test_workload_geometries_and_byte_counts(orc):
    """The workload table holds the stated geometries (28 layers of 2 kv and 12
    query heads at d 128 with layers 0-2 and 25-27 in bf16; 43 MQA layers of
    64 query heads at d 512 over 65,280 packed + 256 dense tokens; ...) and
    their record sizes give the stated bytes per token: 52 / 36 (K 3 / V 2
    bits at d 128), 260 at d 512 and 4 bits, and 730 MB of records per step
    for the V4-Flash-like cache."""
    C = synth.CONFIGS
    q = C["qwen2_1p5b_ctx2048"]
    assert (q["L"], q["Hkv"], q["Hq"], q["d"], q["ctx"], q["kb"], q["vb"]) == (28, 2, 12, 128, 2048, 3, 2)
    assert q["dense_layers"] == (0, 1, 2, 25, 26, 27)
    v = C["v4flash_mqa_ctx65536"]
    assert (v["L"], v["Hkv"], v["Hq"], v["d"], v["ctx"], v["tail"], v["kb"], v["shared_kv"]) == \
        (43, 1, 64, 512, 65536, 256, 4, True)
    assert (v["ctx"] - v["tail"]) % 128 == 0 and (v["ctx"] - v["tail"]) == 65280
    b = C["batched_b32_ctx32768"]
    assert (b["L"], b["B"], b["Hkv"], b["Hq"], b["ctx"], b["kb"], b["vb"], b["T"]) == \
        (32, 32, 8, 32, 32768, 4, 3, 2.0)
    lc = C["longctx_b4_ctx262144"]
    assert (lc["L"], lc["B"], lc["ctx"], lc["tail"]) == (8, 4, 262144, 1024)
    per_tok = lambda d, bits: orc.Codec(d=d, bits=bits).record_bytes // 128
    assert (per_tok(128, 3), per_tok(128, 2), per_tok(512, 4)) == (52, 36, 260)
    assert v["L"] * 65280 * per_tok(512, 4) == 729_830_400
