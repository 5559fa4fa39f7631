"""The encoders' decision-cell quantiser (3- and 4-bit codes).  With z = 128 y
(y the normalised rotated coordinate, |y| <= 1) and cell i = rint(z) + 128
covering z in [i - 128.5, i - 127.5), each cell keeps the count of Lloyd-Max
boundaries below it and the boundary inside it (if any); the code is
count + (z > that boundary).  This equals #{k : y > t_k} exactly only if no
cell holds two boundaries.  Checked here on the f32 tables of every head dim
and bit width, and the lookup replayed in f32 against the direct count on
values spread over [-1, 1] and placed on and next to every boundary."""
import numpy as np
import pytest

SCALE = np.float32(128.0)


def cell_table(t):
    """(count below, boundary x 128 or +huge) for the 257 cells that |y| <= 1 reaches."""
    below = np.zeros(257, np.int32)
    inside = np.full(257, np.float32(3.0e38))
    for i in range(257):
        lo = (np.float32(i - 128) - np.float32(0.5)) / SCALE
        hi = (np.float32(i - 128) + np.float32(0.5)) / SCALE
        below[i] = int(np.sum(t < lo))
        ins = t[(t >= lo) & (t < hi)]
        assert len(ins) <= 1, f"cell {i} holds {len(ins)} boundaries"
        if len(ins):
            inside[i] = ins[0] * SCALE
    return below, inside


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [3, 4])
def test_cells_hold_at_most_one_boundary_and_give_the_count(orc, d, bits):
    t = orc.codebook_f32(bits, d)[1].astype(np.float32)
    below, inside = cell_table(t)
    # the closest pair (b = 4, around 0 at d = 512) is still more than one cell apart
    assert np.min(np.diff(t)) * 128 > 1.0
    rng = np.random.default_rng(bits * 1000 + d)
    y = rng.uniform(-1, 1, 200_000).astype(np.float32)
    near = np.concatenate([t, np.nextafter(t, np.float32(2)), np.nextafter(t, np.float32(-2))])
    edges = (np.arange(-128, 129, dtype=np.float32) + np.float32(0.5)) / SCALE   # cell edges, ties of rint
    y = np.concatenate([y, near, edges, -edges, np.float32([0.0, -0.0, 1.0, -1.0])]).astype(np.float32)
    z = y * SCALE                                   # exact (a power of two)
    i = np.rint(z).astype(np.int64) + 128           # round half to even, as the kernels' conversion
    code = below[i] + (z > inside[i])
    want = np.sum(y[:, None] > t[None, :], axis=1)
    assert np.array_equal(code, want)
