"""Why the tensor-core attention kernels split every f16 operand into hi + lo:
a numpy model of their arithmetic against fp64, on random codes with the
configs' shapes.

The model follows the kernels step by step: centroids enter x 2^16 and each
head's rotated query x 2^s (largest entry near 2^14); scores are
K~hi.q~hi + K~hi.q~lo + K~lo.q~hi (f16 x f16 products are exact in f32) with
f32 accumulation; logits = score . n_K . scale . log2(e) . 2^-(16+s); p =
exp2(t - max); P' = p . n_V . 2^kx (largest near 2^15); values accumulate
V~hi.P'hi + V~hi.P'lo + V~lo.P'hi; the output is brought back by the
orthonormal Hadamard transform.  The "single" variant uses one f16 product
per contraction.  The split stays orders of magnitude inside the 2e-3 bar;
single f16 operands do not meet it.  No oracle arithmetic is used: the
oracle only supplies the Lloyd-Max tables."""
import numpy as np
import pytest
import scipy.linalg

LOG2E = 1.4426950408889634
TOL = 2e-3

# (head dim, query heads per kv head, tokens, K bits, V bits, log-normal sigma of the norms, scale, seed)
CASES = {
    "qwen2_like": (128, 6, 2048, 3, 2, 0.0, 1.0, 0),
    "qwen2_like_peaky": (128, 6, 2048, 3, 2, 0.0, 4.0, 1),
    "v4flash_like": (512, 64, 2048, 4, 4, 0.3, 1.0, 2),
    "batched_like": (128, 4, 4096, 4, 3, 0.0, 1.0, 3),
    "d64_mixed": (64, 8, 2048, 2, 4, 0.5, 2.0, 4),
}


def _f16(x):
    return x.astype(np.float16).astype(np.float32)


def _split(x):
    hi = _f16(x)
    return hi, _f16(x - hi)


def _pow2(e):
    return np.ldexp(np.float32(1.0), e).astype(np.float32)


def _model(qt, kv, kn, vv, vn, scale, split):
    K = (kv * np.float32(2.0 ** 16)).astype(np.float32)
    s = (14 - np.floor(np.log2(np.abs(qt).max(1)))).astype(int)
    Q = (qt * _pow2(s)[:, None]).astype(np.float32)
    if split:
        (Kh, Kl), (Qh, Ql) = _split(K), _split(Q)
        acc = Kh @ Qh.T + Kh @ Ql.T + Kl @ Qh.T
    else:
        acc = _f16(K) @ _f16(Q).T
    t = (acc * kn[:, None] * np.float32(scale * LOG2E) * _pow2(-(16 + s))[None, :]).astype(np.float32)
    p = np.exp2(t - t.max(0)).astype(np.float32)
    l = p.sum(0, dtype=np.float32)
    kx = int(15 - np.ceil(np.log2(vn.max())))
    P = (p * vn[:, None] * _pow2(kx)).astype(np.float32)
    V = (vv * np.float32(2.0 ** 16)).astype(np.float32)
    if split:
        (Vh, Vl), (Ph, Pl) = _split(V), _split(P)
        O = Vh.T @ Ph + Vh.T @ Pl + Vl.T @ Ph
    else:
        O = _f16(V).T @ _f16(P)
    return (O * _pow2(-(16 + kx)) / l).astype(np.float64)


def _fp64(qt, kv, kn, vv, vn, scale):
    t = scale * (kv.astype(np.float64) * kn[:, None]) @ qt.astype(np.float64).T
    p = np.exp(t - t.max(0))
    p /= p.sum(0)
    return (vv.astype(np.float64) * vn[:, None]).T @ p


def _errors(orc, d, H, n, kb, vb, sigma, scale, seed):
    rng = np.random.default_rng(seed)
    ck = orc.codebook_f32(kb, d)[0].astype(np.float32)
    cv = orc.codebook_f32(vb, d)[0].astype(np.float32)
    kv = ck[rng.integers(0, 1 << kb, (n, d))]
    vv = cv[rng.integers(0, 1 << vb, (n, d))]
    kn = (np.sqrt(d) * np.exp(sigma * rng.standard_normal(n))).astype(np.float32)
    vn = (np.sqrt(d) * np.exp(sigma * rng.standard_normal(n))).astype(np.float32)
    qt = (rng.standard_normal((H, d)) / np.sqrt(d)).astype(np.float32)
    Hd = scipy.linalg.hadamard(d) / np.sqrt(d)
    want = Hd @ _fp64(qt, kv, kn, vv, vn, scale)
    return tuple(float(np.abs(Hd @ _model(qt, kv, kn, vv, vn, scale, split) - want).max())
                 for split in (True, False))


@pytest.fixture(scope="module")
def errors(orc):
    return {name: _errors(orc, *args) for name, args in CASES.items()}


@pytest.mark.parametrize("name", sorted(CASES))
def test_hilo_split_is_far_inside_the_tolerance(errors, name):
    assert errors[name][0] <= TOL / 20, errors[name]


def test_single_f16_operands_miss_the_tolerance(errors):
    worst = max(single for _, single in errors.values())
    assert worst > TOL, errors
    assert errors["v4flash_like"][1] > TOL


def _model_terms(qt, kv, kn, vv, vn, scale, score_terms, value_terms):
    """_model with a chosen subset of the three split products per contraction:
    'hh', 'hl' (hi . lo of the second operand), 'lh' (lo of the first . hi)."""
    K = (kv * np.float32(2.0 ** 16)).astype(np.float32)
    s = (14 - np.floor(np.log2(np.abs(qt).max(1)))).astype(int)
    Q = (qt * _pow2(s)[:, None]).astype(np.float32)
    (Kh, Kl), (Qh, Ql) = _split(K), _split(Q)
    prod = {"hh": lambda: Kh @ Qh.T, "hl": lambda: Kh @ Ql.T, "lh": lambda: Kl @ Qh.T}
    acc = sum(prod[t]() for t in score_terms)
    t = (acc * kn[:, None] * np.float32(scale * LOG2E) * _pow2(-(16 + s))[None, :]).astype(np.float32)
    p = np.exp2(t - t.max(0)).astype(np.float32)
    l = p.sum(0, dtype=np.float32)
    kx = int(15 - np.ceil(np.log2(vn.max())))
    P = (p * vn[:, None] * _pow2(kx)).astype(np.float32)
    V = (vv * np.float32(2.0 ** 16)).astype(np.float32)
    (Vh, Vl), (Ph, Pl) = _split(V), _split(P)
    vprod = {"hh": lambda: Vh.T @ Ph, "hl": lambda: Vh.T @ Pl, "lh": lambda: Vl.T @ Ph}
    O = sum(vprod[t]() for t in value_terms)
    return (O * _pow2(-(16 + kx)) / l).astype(np.float64)


@pytest.mark.parametrize("drop", ["score hl", "score lh", "value hl", "value lh"])
def test_no_two_product_split_holds_on_peaky_v4flash_draws(orc, drop):
    """Dropping any one of the three products (in the scores or in the values)
    misses the 2e-3 bar on a V4-Flash-like draw with logits scaled 8x, while
    the three-product split stays far inside it: the tcgen05 kernel's MMA work
    cannot be cut by a third without giving up the tolerance."""
    d, H, n, kb, vb, sigma, scale, seed = 512, 64, 2048, 4, 4, 0.3, 8.0, 6
    rng = np.random.default_rng(seed)
    ck = orc.codebook_f32(kb, d)[0].astype(np.float32)
    cv = orc.codebook_f32(vb, d)[0].astype(np.float32)
    kv = ck[rng.integers(0, 1 << kb, (n, d))]
    vv = cv[rng.integers(0, 1 << vb, (n, d))]
    kn = (np.sqrt(d) * np.exp(sigma * rng.standard_normal(n))).astype(np.float32)
    vn = (np.sqrt(d) * np.exp(sigma * rng.standard_normal(n))).astype(np.float32)
    qt = (rng.standard_normal((H, d)) / np.sqrt(d)).astype(np.float32)
    Hd = scipy.linalg.hadamard(d) / np.sqrt(d)
    want = Hd @ _fp64(qt, kv, kn, vv, vn, scale)
    full = ("hh", "hl", "lh")
    kind, term = drop.split()
    st = tuple(t for t in full if not (kind == "score" and t == term))
    vt = tuple(t for t in full if not (kind == "value" and t == term))
    err = float(np.abs(Hd @ _model_terms(qt, kv, kn, vv, vn, scale, st, vt) - want).max())
    err3 = float(np.abs(Hd @ _model_terms(qt, kv, kn, vv, vn, scale, full, full) - want).max())
    assert err3 <= TOL / 20
    assert err > TOL, (drop, err)
