"""Pins for the oracle's decode attention and chunked-eviction bookkeeping."""
import numpy as np
import pytest
import torch

import synth


def _codec(orc, d, bits, T=0.0):
    return orc.Codec(d=d, bits=bits, seed=1, T=T)


def test_dense_matches_torch_sdpa(orc):
    """Plain softmax attention in fp64 equals torch's scaled_dot_product_attention
    (CPU, float64) -- the textbook routine."""
    rng = np.random.default_rng(0)
    G, n, d = 6, 37, 128
    q, K, V = rng.standard_normal((G, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    scale = 0.3
    got = orc.attention(q, K, V, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).reshape(1, G, 1, d),
        torch.from_numpy(K)[None, None].expand(1, G, n, d),
        torch.from_numpy(V)[None, None].expand(1, G, n, d), scale=scale)[0, :, 0, :].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_special_cases(orc):
    rng = np.random.default_rng(1)
    d = 64
    V = rng.standard_normal((9, d))
    K = rng.standard_normal((9, d))
    # one token: the output is that value
    np.testing.assert_allclose(orc.attention(rng.standard_normal((2, d)), K[:1], V[:1], 1.0),
                               np.repeat(V[:1], 2, 0), atol=1e-15)
    # q = 0: the mean of the values
    np.testing.assert_allclose(orc.attention(np.zeros((1, d)), K, V, 1.0)[0], V.mean(0), atol=1e-14)
    # identical tokens: that value
    np.testing.assert_allclose(orc.attention(rng.standard_normal((1, d)), np.repeat(K[:1], 5, 0),
                                             np.repeat(V[:1], 5, 0), 0.7)[0], V[0], atol=1e-14)
    # empty context: zero output
    assert np.all(orc.attention(np.ones((1, d)), K[:0], V[:0], 1.0) == 0)


def test_compressed_one_token_returns_decoded_value(orc):
    d = 128
    ck, cv = _codec(orc, d, 3), _codec(orc, d, 2)
    kx, vx = synth.gaussian_bf16((1, d), 1), synth.gaussian_bf16((1, d), 2)
    kr, vr = orc.encode_records(kx, ck), orc.encode_records(vx, cv)
    q = synth.gaussian_bf16((4, d), 3)
    out = orc.unit_attention(q, ck, cv, kr, vr, 1, None, None, 1.0)
    np.testing.assert_allclose(out, np.repeat(orc.decode_records(vr, 1, cv), 4, 0), atol=1e-14)


@pytest.mark.parametrize("T", [0.0, 2.0])
def test_rotated_form_equals_brute_force(orc, T):
    """Scoring against q~ = H(s q)/sqrt(d) with n * yhat and one inverse transform
    of the value accumulator equals attention over fully decoded vectors."""
    d, nc, nd, G = 128, 300, 40, 6
    ck, cv = _codec(orc, d, 4, T), _codec(orc, d, 3, T)
    k = synth.gaussian_bf16((nc, d), 4, outlier_frac=0.02)
    v = synth.gaussian_bf16((nc, d), 5)
    kr, vr = orc.encode_records(k, ck), orc.encode_records(v, cv)
    kd, vd = synth.gaussian_bf16((nd, d), 6), synth.gaussian_bf16((nd, d), 7)
    q = synth.gaussian_bf16((G, d), 8, scale=1 / np.sqrt(d))
    brute = orc.unit_attention(q, ck, cv, kr, vr, nc, kd, vd, 1.0)
    rot = orc.attention_rotated(orc.bf16_to_f64(q),
                                orc.decode_records(kr, nc, ck, rotated=True),
                                orc.decode_records(vr, nc, cv, rotated=True),
                                orc.bf16_to_f64(kd), orc.bf16_to_f64(vd), 1.0,
                                orc.signs(1, d), orc.signs(1, d))
    np.testing.assert_allclose(rot, brute, atol=1e-12)


def test_query_head_permutation_permutes_outputs(orc):
    d = 64
    ck = _codec(orc, d, 3)
    kr = orc.encode_records(synth.gaussian_bf16((50, d), 1), ck)
    vr = orc.encode_records(synth.gaussian_bf16((50, d), 2), ck)
    q = synth.gaussian_bf16((4, d), 3)
    perm = np.array([2, 0, 3, 1])
    a = orc.unit_attention(q, ck, ck, kr, vr, 50, None, None, 0.5)
    b = orc.unit_attention(q[perm], ck, ck, kr, vr, 50, None, None, 0.5)
    np.testing.assert_allclose(b, a[perm], atol=0)


def test_softcap_closed_form_position(orc):
    """Soft cap after the scale multiply (arc PR #98, softcapping fix): with
    cap 2 and scaled logits 2 atanh(1/2) and -2 atanh(1/2) the capped logits
    are exactly +1 and -1, so one-hot values return the weights
    1/(1 + e^-2) and 1/(1 + e^2).  Capping before the scale (scale 1/2 here)
    or not at all gives other weights."""
    d, cap, scale = 64, 2.0, 0.5
    a = 2 * np.arctanh(0.5) / scale          # q.k of token 0
    q = np.zeros((1, d)); q[0, 0] = 1.0
    K = np.zeros((2, d)); K[0, 0], K[1, 0] = a, -a
    V = np.zeros((2, d)); V[0, 3] = V[1, 7] = 1.0
    out = orc.attention(q, K, V, scale, cap)[0]
    w0 = 1.0 / (1.0 + np.exp(-2.0))
    assert abs(out[3] - w0) < 1e-14 and abs(out[7] - (1.0 - w0)) < 1e-14
    assert abs(orc.attention(q, K, V, scale)[0, 3] - w0) > 0.01        # uncapped: 0.900


def test_softcap_bounds_the_weight_ratio(orc):
    """Capped logits lie in (-cap, cap), so no two softmax weights differ by
    more than a factor e^(2 cap), however large the raw logits are."""
    rng = np.random.default_rng(5)
    d, n, cap = 40, 40, 1.5
    q = rng.standard_normal((3, d)) * 10
    K = rng.standard_normal((n, d)) * 10
    V = np.zeros((n, n)); np.fill_diagonal(V, 1.0)        # one-hot rows: out = weights
    w = orc.attention(q, K, V, 1.0, cap)
    assert np.all(w.max(1) / w.min(1) <= np.exp(2 * cap) * (1 + 1e-12))
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-14)
    raw = orc.attention(q, K, V, 1.0)
    assert np.all(raw.max(1) > 1e6 * raw.min(1))          # the cap is what bounds it


def test_softcap_large_cap_is_no_cap(orc):
    """cap * tanh(s / cap) -> s as cap -> infinity."""
    rng = np.random.default_rng(6)
    q, K, V = rng.standard_normal((4, 64)), rng.standard_normal((20, 64)), rng.standard_normal((20, 64))
    np.testing.assert_allclose(orc.attention(q, K, V, 0.3, 1e7), orc.attention(q, K, V, 0.3), atol=1e-11)


def test_softcap_rotated_form_equals_brute_force(orc):
    d, nc, nd, G = 64, 200, 30, 4
    ck, cv = _codec(orc, d, 3), _codec(orc, d, 2)
    k, v = synth.gaussian_bf16((nc, d), 14), synth.gaussian_bf16((nc, d), 15)
    kr, vr = orc.encode_records(k, ck), orc.encode_records(v, cv)
    kd, vd = synth.gaussian_bf16((nd, d), 16), synth.gaussian_bf16((nd, d), 17)
    q = synth.gaussian_bf16((G, d), 18)
    brute = orc.unit_attention(q, ck, cv, kr, vr, nc, kd, vd, 0.5, softcap=3.0)
    rot = orc.attention_rotated(orc.bf16_to_f64(q), orc.decode_records(kr, nc, ck, rotated=True),
                                orc.decode_records(vr, nc, cv, rotated=True),
                                orc.bf16_to_f64(kd), orc.bf16_to_f64(vd), 0.5,
                                orc.signs(1, d), orc.signs(1, d), softcap=3.0)
    np.testing.assert_allclose(rot, brute, atol=1e-12)
    assert np.max(np.abs(brute - orc.unit_attention(q, ck, cv, kr, vr, nc, kd, vd, 0.5))) > 1e-2


# --------------------------------------------------------------------------- eviction


def test_retention_floor_each_term_binds(orc):
    """window + max(t_q - 1, margin) (arc PR #98, "Mutation runs": each term is
    tested where it binds)."""
    assert orc.retention_floor(128, 1, 16) == 144         # margin binds
    assert orc.retention_floor(128, 40, 16) == 167        # t_q - 1 binds
    assert orc.retention_floor(0, 1, 16) == 16            # window term
    assert orc.retention_floor(64, 17, 16) == 80          # equal terms
    assert orc.chunks_to_evict(271, 128, 1, 16) == 0
    assert orc.chunks_to_evict(272, 128, 1, 16) == 1      # reaches the bound
    assert orc.chunks_to_evict(144 + 256, 128, 1, 16) == 2
    assert orc.chunks_to_evict(144 + 255, 128, 1, 16) == 1


def test_tail_bound_over_a_long_decode(orc):
    """Appending 65,536 tokens one at a time with chunked eviction leaves 510
    records and a 256-token tail, and the tail never exceeds 272."""
    length, n_chunks, hi = 0, 0, 0
    for _ in range(65536):
        length += 1
        hi = max(hi, length)
        k = orc.chunks_to_evict(length, 128, 1, 16)
        length -= 128 * k
        n_chunks += k
    assert (n_chunks, length) == (510, 256) and hi == 272


def test_eviction_is_append_only_and_tail_exact(orc):
    """Later evictions leave earlier records byte-identical, and the tokens
    still in the tail are the dense tokens themselves."""
    d, cap, Hkv = 64, 272, 2
    ck = _codec(orc, d, 4)
    toks = synth.gaussian_bf16((Hkv, 600, d), 12)
    ring = np.zeros((Hkv, cap, d), np.uint16)
    krec = np.zeros((Hkv, 8, ck.record_bytes), np.uint8)
    start = length = n_chunks = 0
    snapshots = []
    for t in range(600):
        ring[:, (start + length) % cap] = toks[:, t]
        length += 1
        start, length, nc = orc.evict(ring, ring, start, length, n_chunks, krec, None, ck, None,
                                      128, 1, 16)
        if nc != n_chunks:
            snapshots.append(krec.copy())
            n_chunks = nc
    assert n_chunks == 3 and length == 600 - 384
    for i, (a, b) in enumerate(zip(snapshots, snapshots[1:])):
        np.testing.assert_array_equal(a[:, :i + 1], b[:, :i + 1])
    # record r holds tokens [128 r, 128 r + 128)
    for r in range(3):
        np.testing.assert_array_equal(krec[:, r], np.stack(
            [orc.encode_records(toks[h, 128 * r:128 * r + 128], ck)[0] for h in range(Hkv)]))
    tail = ring[:, (start + np.arange(length)) % cap]
    np.testing.assert_array_equal(tail, toks[:, 384:600])
