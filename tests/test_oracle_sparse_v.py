"""Pins of the oracle's sparse-V attention (turboquant_plus commit log,
"safer-asym + sparse-V dequant": the value work of tokens whose post-softmax
weight is negligible is skipped).  The skip rule is this project's reading
(a block of tokens is skipped for a group of query heads when every logit of
the group in the block is below the running maximum of the blocks visited
before plus ln eps); it is pinned by hand-worked cases and by the error bound
it implies, eps * (skipped tokens) * max |v| against exact attention."""
import math

import numpy as np
import pytest


def _kv(logits, d=2):
    """Keys giving the logits for q = e_0, values = distinct rows."""
    n = len(logits)
    K = np.zeros((n, d))
    K[:, 0] = logits
    V = np.arange(n * d, dtype=np.float64).reshape(n, d) + 1.0
    return K, V


def test_second_block_below_threshold_is_skipped(orc):
    K, V = _kv([0.0, 0.0, -20.0, -21.0])
    q = np.array([[1.0, 0.0]])
    blocks = [(0, 2, 0), (2, 4, 0)]
    out, sk = orc.attention_sparse_v(q, K, V, 1.0, math.exp(-10), 1, blocks)
    Z = 2 + math.exp(-20) + math.exp(-21)
    np.testing.assert_allclose(out[0], (V[0] + V[1]) / Z, rtol=1e-15)
    assert sk == 2
    # visited first, the low block has no maximum to compare with: nothing skipped
    out2, sk2 = orc.attention_sparse_v(q, K, V, 1.0, math.exp(-10), 1, [(2, 4, 0), (0, 2, 0)])
    np.testing.assert_allclose(out2, orc.attention(q, K, V, 1.0), rtol=1e-15)
    assert sk2 == 0
    # in separate sequences the maxima are not shared: nothing skipped
    assert orc.attention_sparse_v(q, K, V, 1.0, math.exp(-10), 1, [(0, 2, 0), (2, 4, 1)])[1] == 0


def test_threshold_is_strict_and_eps_zero_is_exact(orc):
    K, V = _kv([0.0, -10.0])
    q = np.array([[1.0, 0.0]])
    blocks = [(0, 1, 0), (1, 2, 0)]
    # logit -10 against 0 + ln(e^-10): not strictly below, kept
    assert orc.attention_sparse_v(q, K, V, 1.0, math.exp(-10) * (1 - 1e-12), 1, blocks)[1] == 0
    assert orc.attention_sparse_v(q, K, V, 1.0, math.exp(-10) * (1 + 1e-9), 1, blocks)[1] == 1
    out, sk = orc.attention_sparse_v(q, K, V, 1.0, 0.0, 1, blocks)
    assert sk == 0
    np.testing.assert_allclose(out, orc.attention(q, K, V, 1.0), rtol=1e-15)


def test_a_group_skips_only_when_every_head_is_low(orc):
    """Head 0 sees the second block far below its maximum, head 1 sees it as
    its maximum: skipped for head 0 alone in groups of one, kept for both in a
    group of two."""
    K = np.array([[10.0, 0.0], [-10.0, 5.0]])
    V = np.array([[1.0, 2.0], [3.0, 4.0]])
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    blocks = [(0, 1, 0), (1, 2, 0)]
    out1, sk1 = orc.attention_sparse_v(q, K, V, 1.0, 1e-3, 1, blocks)
    assert sk1 == 1
    np.testing.assert_allclose(out1[0], V[0] / (1 + math.exp(-20)), rtol=1e-15)
    np.testing.assert_allclose(out1[1], orc.attention(q[1:], K, V, 1.0)[0], rtol=1e-15)
    out2, sk2 = orc.attention_sparse_v(q, K, V, 1.0, 1e-3, 2, blocks)
    assert sk2 == 0
    np.testing.assert_allclose(out2, orc.attention(q, K, V, 1.0), rtol=1e-15)


@pytest.mark.parametrize("eps", [1e-3, 1e-6])
def test_error_bound_on_peaky_logits(orc, eps):
    """Against exact attention every output coordinate is within
    eps * (skipped tokens of the head's group) * max |v|, since a skipped token's
    weight relative to the final maximum is below eps and the denominator is
    at least 1; on these peaky logits most blocks are skipped."""
    rng = np.random.default_rng(5)
    n, d, G = 16 * 128, 16, 4
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    q = rng.standard_normal((G, d))
    blocks = orc.sparse_v_blocks(n // 128, 4)
    # a dominant key (an attention sink, logit 60 or more for every head) opens every sequence
    u = q.sum(0)
    sink = u * (60.0 / np.min(q @ u))
    for b in blocks:
        if b[0] % 128 == 32 * (b[2] % 4) and (b[0] // 128) % 4 == 0:
            K[b[0]] = sink
    out, sk = orc.attention_sparse_v(q, K, V, 1.0, eps, G, blocks)
    exact = orc.attention(q, K, V, 1.0)
    assert sk > n // 2
    assert np.max(np.abs(out - exact)) <= eps * sk * np.max(np.abs(V))


def test_schedule_blocks(orc):
    """Split s, warp w: tokens 32 w .. 32 w + 31 of the split's records, one
    sequence per (split, warp), records in order."""
    b = orc.sparse_v_blocks(5, 2)
    assert len(b) == 5 * 4
    assert b[:3] == [(0, 32, 0), (128, 160, 0), (32, 64, 1)]
    assert (4 * 128 + 96, 4 * 128 + 128, 2 * 4 + 3) in b
    assert sorted(t for bb in b for t in range(bb[0], bb[1])) == list(range(5 * 128))


def test_schedule_blocks_of_grouped_ctas(orc):
    """Three 4-warp groups per CTA: split s deals its records out round robin,
    group g visiting records g, g + 3, ... of the split; one sequence per
    (split, group, warp)."""
    b = orc.sparse_v_blocks(7, 5, groups=3)
    assert len(b) == 7 * 4
    seq = {}
    for lo, hi, s in b:
        seq.setdefault(s, []).append(lo // 128)
    # split 0 (records 0-4): group 0 takes 0 and 3, group 1 takes 1 and 4, group 2 takes 2
    assert seq[0 * 4 + 1] == [0, 3] and seq[1 * 4 + 2] == [1, 4] and seq[2 * 4 + 0] == [2]
    # split 1 (records 5, 6): groups 0 and 1 take one record each, group 2 none
    assert seq[(3 + 0) * 4 + 3] == [5] and seq[(3 + 1) * 4 + 0] == [6] and (3 + 2) * 4 not in seq
    assert b[0] == (0, 32, 0) and (3 * 128 + 32, 3 * 128 + 64, 1) in b
    assert sorted(t for bb in b for t in range(bb[0], bb[1])) == list(range(7 * 128))
    assert orc.sparse_v_blocks(5, 2, groups=1) == orc.sparse_v_blocks(5, 2)
