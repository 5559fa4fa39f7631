"""The encoders' decision-cell quantiser (2-, 3- and 4-bit codes).  With z = 128 y
(y the normalised rotated coordinate, |y| <= 1) and cell i = rint(z) + 128
covering z in [i - 128.5, i - 127.5), each cell keeps the count of Lloyd-Max
boundaries below it and the boundary inside it (if any); the code is
count + (z > that boundary).  This equals #{k : y > t_k} exactly only if no
cell holds two boundaries.  Checked here on the f32 tables of every head dim
and bit width, and the lookup replayed in f32 against the direct count on
values spread over [-1, 1] and placed on and next to every boundary.  The
d-128 tensor-core encoder uses cells moved down by 2^-8 (index = bits 7..15
of the f32 sum z + 2^16 + 128.5, which rounds z + 128.5 to the 2^-7 grid):
the same checks, plus values on and next to those cells' edges."""
import numpy as np
import pytest

SCALE = np.float32(128.0)


SHIFT = np.float32(2.0 ** -8)
MAGIC_SHIFTED = np.float32(65664.5)   # 2^16 + 128.5


def cell_table(t, shifted=False):
    """(count below, boundary x 128 or +huge) for the 257 cells that |y| <= 1 reaches."""
    below = np.zeros(257, np.int32)
    inside = np.full(257, np.float32(3.0e38))
    sh = SHIFT if shifted else np.float32(0)
    for i in range(257):
        lo = (np.float32(i - 128) - np.float32(0.5) - sh) / SCALE
        hi = (np.float32(i - 128) + np.float32(0.5) - sh) / SCALE
        below[i] = int(np.sum(t < lo))
        ins = t[(t >= lo) & (t < hi)]
        assert len(ins) <= 1, f"cell {i} holds {len(ins)} boundaries"
        if len(ins):
            inside[i] = ins[0] * SCALE
    return below, inside


def cell_index(z, shifted):
    if not shifted:
        return np.rint(z).astype(np.int64) + 128       # round half to even, as the kernels' conversion
    u = (z.astype(np.float32) + MAGIC_SHIFTED).astype(np.float32)   # one f32 add, rounded to nearest even
    return ((u.view(np.uint32) >> 7) & 0x1FF).astype(np.int64)


@pytest.mark.parametrize("shifted", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_cells_hold_at_most_one_boundary_and_give_the_count(orc, d, bits, shifted):
    t = orc.codebook_f32(bits, d)[1].astype(np.float32)
    below, inside = cell_table(t, shifted)
    # the closest pair (b = 4, around 0 at d = 512) is still more than one cell apart
    assert np.min(np.diff(t)) * 128 > 1.0
    rng = np.random.default_rng(bits * 1000 + d)
    y = rng.uniform(-1, 1, 200_000).astype(np.float32)
    near = np.concatenate([t, np.nextafter(t, np.float32(2)), np.nextafter(t, np.float32(-2))])
    edges = (np.arange(-128, 129, dtype=np.float32) + np.float32(0.5)) / SCALE   # cell edges, ties of rint
    if shifted:
        edges = (edges * SCALE - SHIFT) / SCALE     # exact: multiples of 2^-8 below 2^8
    edges = np.concatenate([edges, np.nextafter(edges, np.float32(2)), np.nextafter(edges, np.float32(-2))])
    y = np.concatenate([y, near, edges, -edges, np.float32([0.0, -0.0, 1.0, -1.0])]).astype(np.float32)
    y = y[np.abs(y) <= 1]                           # a normalised coordinate
    z = y * SCALE                                   # exact (a power of two)
    i = cell_index(z, shifted)
    assert i.min() >= 0 and i.max() <= 256
    code = below[i] + (z > inside[i])
    want = np.sum(y[:, None] > t[None, :], axis=1)
    assert np.array_equal(code, want)
