"""Pins of the oracle's rollback ("feat(v4): TurboQuant KV storage for
DeepSeek-V4", "What landed": the cache reports its length in tokens and maps
truncation onto both time bases -- the packed records and the dense tail --,
and a deep rollback into the packed region has to dequantise)."""
import math

import numpy as np
import pytest

import synth


@pytest.mark.parametrize("n,length", [(0, 0), (0, 77), (3, 0), (3, 200), (5, 143)])
def test_span_stays_total(orc, n, length):
    """For every target length T the rolled-back stream holds exactly
    min(max(T, 0), 128 n + len) tokens, the records never grow, the tail
    stays below 128 tokens after a rollback into the records, and the tail
    start is reset exactly when records are dropped."""
    total = 128 * n + length
    for T in range(-2, total + 3):
        n2, len2, reset, m = orc.rollback_counts(n, length, T)
        want = min(max(T, 0), total)
        assert 128 * n2 + len2 == want
        assert n2 <= n
        assert reset == (want < 128 * n)
        if reset:
            assert len2 < 128 and m == len2 and n2 == want // 128
        else:
            assert (n2, m) == (n, 0)


def test_rollback_then_regrow_restores_the_counters(orc):
    """A deep rollback followed by re-appending the same tokens and evicting
    (max 2 chunks a call) returns to the original record count and tail
    length: the two time bases stay consistent through truncation."""
    window, t_q, margin = 128, 1, 16
    floor_ = orc.retention_floor(window, t_q, margin)
    for T0, T in ((1000, 700), (1000, 300), (1000, 256), (900, 899), (1000, 0)):
        n = max(0, (T0 - floor_) // 128)
        ln = T0 - 128 * n
        n2, len2, _, _ = orc.rollback_counts(n, ln, T)
        while 128 * n2 + len2 < T0:              # append one token at a time, evicting as the bound is hit
            len2 += 1
            k = min(orc.chunks_to_evict(len2, window, t_q, margin), 2)
            n2, len2 = n2 + k, len2 - 128 * k
        assert (n2, len2) == (n, ln), (T0, T)


def test_deep_rollback_of_a_spike_record(orc):
    """Tokens whose codes are all k decode to one spike n * s_0 * c_k * sqrt(d)
    at coordinate 0 (H of a constant vector is a multiple of e_0); a deep
    rollback that keeps 5 such tokens writes bf16 of that value there and
    zeros elsewhere, and leaves the tail start at 0."""
    d, bits = 64, 3
    cod = orc.Codec(d=d, bits=bits)
    c, _, s = cod.tables()
    enc = {"codes": np.full((128, d), 6, np.uint8), "norms": np.linspace(0.5, 3.0, 128).astype(np.float32),
           "is_out": np.zeros((128, d), np.uint8), "oval": np.zeros((128, d), np.uint16)}
    rec = orc.pack_records(enc, cod)                                 # one record
    recs = np.stack([np.zeros_like(rec[0]), rec[0]])[None]            # [Hkv=1, 2 records, bytes]
    tail = np.full((1, 272, d), 0x7FC0, np.uint16)                    # stale ring contents
    start, length, n = orc.rollback(tail, None, 40, 100, 2, recs, None, cod, None, 128 + 5)
    assert (start, length, n) == (0, 5, 1)
    for i in range(5):
        spike = float(enc["norms"][i]) * s[0] * float(c[6]) * math.sqrt(d)
        assert tail[0, i, 0] == orc.f64_to_bf16(spike)
        assert np.all(tail[0, i, 1:] & 0x7FFF == 0)                    # zeros (of either sign)
    assert np.all(tail[0, 5:] == 0x7FC0)                              # slots past the kept tokens untouched


def test_rollback_within_the_tail_keeps_the_ring(orc):
    d, bits = 64, 2
    cod = orc.Codec(d=d, bits=bits)
    tail = synth.gaussian_bf16((2, 272, d), 3)
    before = tail.copy()
    recs = np.zeros((2, 4, cod.record_bytes), np.uint8)
    assert orc.rollback(tail, tail, 17, 150, 3, recs, recs, cod, cod, 3 * 128 + 90) == (17, 90, 3)
    np.testing.assert_array_equal(tail, before)
    assert orc.rollback(tail, tail, 17, 150, 3, recs, recs, cod, cod, 10 ** 6) == (17, 150, 3)
