"""GPU parity of the fused decode attention (tq_decode_attn) against the
oracle's brute-force softmax attention over fully dequantised vectors.

Two comparisons per case: (1) the oracle attends the GPU's own records (this
isolates the attention numerics, bar 2e-3 max-abs), (2) end to end, the oracle
encodes the same inputs itself and attends its own records (bar 2e-3 too;
boundary-band code flips are the only other difference)."""
import math

import numpy as np
import pytest

import synth
import tq_testlib as tl

pytestmark = pytest.mark.gpu
TOL = 2e-3


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


def run_case(tq, orc, *, d, G, Hkv, B, L, chunks, tails, kb, vb, T=0.0, shared=False, dense=False,
             tail_cap=None, splits=0, seed=0, q_pad=0, k_outlier_frac=0.0, end_to_end=True, scale=1.0,
             cuda_core_path=False, zero_every=0, softcap=0.0, oracle_softcap=None):
    """chunks[b], tails[b]: compressed records and dense tail tokens of batch b
    (the same for every layer).  softcap: the logit cap of the GPU call and, unless
    oracle_softcap says otherwise, of the oracle.  Returns (gpu_out, oracle_out,
    oracle_e2e_out)."""
    ocap = softcap if oracle_softcap is None else oracle_softcap
    import torch
    dev = "cuda"
    Hq = G * Hkv
    max_chunks = max(chunks) if not dense else 0
    rec_cap = max(max_chunks, 1)
    tail_cap = tail_cap or max(max(tails), 1)
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = kc if shared else tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    okc, ovc = _ocodec(orc, kc), _ocodec(orc, vc)
    ntok = rec_cap * 128
    kx = synth.gaussian_bf16((L, B, Hkv, ntok, d), seed + 1, outlier_frac=k_outlier_frac,
                             lognormal_sigma=0.3)
    vx = kx if shared else synth.gaussian_bf16((L, B, Hkv, ntok, d), seed + 2)
    if zero_every:  # zero-norm tokens (every zero_every-th token of K and of V)
        kx = kx.copy()
        kx[..., ::zero_every, :] = 0
        vx = kx if shared else vx.copy()
        if not shared:
            vx[..., 3::zero_every, :] = 0
    kt = synth.gaussian_bf16((L, B, Hkv, tail_cap, d), seed + 3)
    vt = kt if shared else synth.gaussian_bf16((L, B, Hkv, tail_cap, d), seed + 4)
    qb = synth.gaussian_bf16((L, B, Hq + q_pad, d), seed + 5, scale=1 / math.sqrt(d))
    rng = np.random.default_rng(seed)
    tstart = rng.integers(0, tail_cap, size=(L, B)).astype(np.int32)
    n_chunks = np.tile(np.array(chunks, np.int32), (L, 1))
    tail_len = np.tile(np.array(tails, np.int32), (L, 1))

    q = tl.to_bf16_tensor(qb, dev)[:, :, :Hq, :]          # batch stride (Hq + q_pad) * d
    out = torch.full((L, B, Hq, d), float("nan"), dtype=torch.float32, device=dev)
    kw = dict(q=q, out=out, scale=scale)
    rec_np = {}
    if not dense:
        krec = torch.zeros((L, B, Hkv, rec_cap, kc.record_bytes), dtype=torch.uint8, device=dev)
        tq.tq_encode(kc, tl.to_bf16_tensor(kx, dev).reshape(L * B * Hkv, ntok, d),
                     krec.view(L * B * Hkv, rec_cap, kc.record_bytes))
        if shared:
            vrec = krec
        else:
            vrec = torch.zeros((L, B, Hkv, rec_cap, vc.record_bytes), dtype=torch.uint8, device=dev)
            tq.tq_encode(vc, tl.to_bf16_tensor(vx, dev).reshape(L * B * Hkv, ntok, d),
                         vrec.view(L * B * Hkv, rec_cap, vc.record_bytes))
        kw.update(k_rec=krec, v_rec=vrec, n_chunks=torch.from_numpy(n_chunks).to(dev), max_chunks=max_chunks)
        rec_np["k"], rec_np["v"] = krec.cpu().numpy(), vrec.cpu().numpy()
    if max(tails) > 0:
        kw.update(k_tail=tl.to_bf16_tensor(kt, dev), v_tail=tl.to_bf16_tensor(vt, dev),
                  tail_start=torch.from_numpy(tstart).to(dev), tail_len=torch.from_numpy(tail_len).to(dev),
                  max_tail=max(tails))
    kw["n_kv_heads"] = Hkv
    tq.decode_attn(k_codec=None if dense else kc, v_codec=None if dense else vc, splits=splits,
                   cuda_core_path=cuda_core_path, softcap=softcap, **kw)
    torch.cuda.synchronize()
    got = out.cpu().numpy()

    want = np.zeros_like(got, dtype=np.float64)
    want_e2e = np.zeros_like(want) if (end_to_end and not dense) else None
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                nc = 0 if dense else chunks[b]
                slots = (tstart[l, b] + np.arange(tails[b])) % tail_cap
                kd, vd = kt[l, b, h, slots], vt[l, b, h, slots]
                qh = qb[l, b, h * G:(h + 1) * G]
                kr = rec_np["k"][l, b, h] if not dense else None
                vr = rec_np["v"][l, b, h] if not dense else None
                want[l, b, h * G:(h + 1) * G] = orc.unit_attention(qh, okc, ovc, kr, vr, nc * 128, kd, vd, scale,
                                                                   ocap)
                if want_e2e is not None:
                    okr = orc.encode_records(kx[l, b, h, :nc * 128], okc) if nc else None
                    ovr = orc.encode_records(vx[l, b, h, :nc * 128], ovc) if nc else None
                    want_e2e[l, b, h * G:(h + 1) * G] = orc.unit_attention(qh, okc, ovc, okr, ovr, nc * 128,
                                                                           kd, vd, scale, ocap)
    return got, want, want_e2e


def _assert_close(got, want, tol=TOL):
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - want))
    assert err <= tol, f"max abs err {err}"
    return err


CASES = {
    "tiny_gqa4_tail": dict(d=64, G=4, Hkv=2, B=2, L=2, chunks=[3, 1], tails=[50, 0], kb=3, vb=2),
    "qwen_like_gqa6": dict(d=128, G=6, Hkv=2, B=1, L=2, chunks=[16], tails=[0], kb=3, vb=2),
    "outliers_gqa4": dict(d=128, G=4, Hkv=2, B=2, L=1, chunks=[4, 2], tails=[0, 0], kb=4, vb=3, T=2.0,
                          k_outlier_frac=0.02),
    "mqa_shared_d512": dict(d=512, G=64, Hkv=1, B=1, L=1, chunks=[5], tails=[256], kb=4, vb=4, shared=True,
                            tail_cap=272),
    "d256_mha_b1": dict(d=256, G=1, Hkv=4, B=1, L=1, chunks=[2], tails=[70], kb=1, vb=4),
    "d128_gqa2_b4b1": dict(d=128, G=2, Hkv=2, B=3, L=1, chunks=[2, 0, 3], tails=[10, 64, 0], kb=4, vb=1),
    "gqa8_q_stride": dict(d=128, G=8, Hkv=1, B=2, L=1, chunks=[3, 3], tails=[20, 5], kb=2, vb=3, q_pad=3),
    "gqa3_odd_group": dict(d=64, G=3, Hkv=2, B=1, L=1, chunks=[2], tails=[9], kb=3, vb=3),
    "hot_logits_gqa6": dict(d=128, G=6, Hkv=1, B=1, L=1, chunks=[3], tails=[0], kb=3, vb=2, scale=4.0),
    "outliers_both_d64": dict(d=64, G=8, Hkv=1, B=2, L=1, chunks=[2, 1], tails=[3, 0], kb=2, vb=4, T=1.5,
                              k_outlier_frac=0.05),
}

PATHS = ["automatic", "cuda_core"]  # automatic = tensor cores where the kernel applies


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_cases(tq, orc, name, path):
    got, want, e2e = run_case(tq, orc, cuda_core_path=(path == "cuda_core"), **CASES[name])
    _assert_close(got, want)
    if e2e is not None:
        _assert_close(got, e2e)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kb", [1, 2, 3, 4])
@pytest.mark.parametrize("vb", [1, 2, 3, 4])
def test_tensor_core_bit_widths(tq, orc, d, kb, vb):
    """Every (key bits, value bits) pair of the tensor-core kernel, two records."""
    got, want, _ = run_case(tq, orc, d=d, G=4, Hkv=1, B=1, L=1, chunks=[2], tails=[0], kb=kb, vb=vb,
                            end_to_end=False, seed=kb * 10 + vb)
    _assert_close(got, want)


@pytest.mark.parametrize("kb,vb,G,shared", [(4, 4, 64, True), (2, 3, 4, False), (3, 1, 8, False), (1, 2, 6, False),
                                             (3, 3, 32, False)])
def test_tensor_core_d512(tq, orc, kb, vb, G, shared):
    """Head dim 512 on its mma.sync kernel (8 or 16 query heads per CTA), with
    a dense tail on the general kernel."""
    got, want, _ = run_case(tq, orc, d=512, G=G, Hkv=1, B=1, L=1, chunks=[3], tails=[40], kb=kb, vb=kb if shared else vb,
                            shared=shared, end_to_end=False, seed=kb * 10 + vb + G, cuda_core_path=2)
    _assert_close(got, want)


@pytest.mark.parametrize("kb,vb,G,shared,chunks", [(4, 4, 64, True, [3]), (1, 1, 16, False, [2]),
                                                    (2, 4, 48, False, [2]), (4, 2, 64, False, [4]),
                                                    (3, 3, 64, True, [2]), (3, 2, 32, False, [1]),
                                                    (4, 4, 128, True, [2])])
def test_tcgen05_d512(tq, orc, kb, vb, G, shared, chunks):
    """Head dim 512 with 16-128 query heads per kv head on the tcgen05 kernel
    (64 heads per CTA, scores and outputs in tensor memory); dense tail on the
    general kernel."""
    got, want, _ = run_case(tq, orc, d=512, G=G, Hkv=1, B=1, L=1, chunks=chunks, tails=[40], kb=kb,
                            vb=kb if shared else vb, shared=shared, end_to_end=False, seed=kb * 7 + vb + G)
    _assert_close(got, want)


def test_tcgen05_d512_multi_record_splits(tq, orc):
    """Several records per CTA (the ring's phases wrap, the running max moves
    lazily) on two batches and layers; one split per unit and three splits
    give the same result."""
    cfg = dict(d=512, G=64, Hkv=1, B=2, L=2, chunks=[6, 3], tails=[17, 0], kb=4, vb=4, shared=True,
               end_to_end=False, seed=5)
    a, want, _ = run_case(tq, orc, splits=1, **cfg)
    b, _, _ = run_case(tq, orc, splits=3, **cfg)
    _assert_close(a, want)
    _assert_close(b, want)
    assert np.max(np.abs(a - b)) <= 1e-5


def test_tcgen05_d512_hot_logits_and_zero_tokens(tq, orc):
    """Peaky softmax (scale 8: the running max moves, lazily, several times in
    one split of six records) over a cache with zero-norm tokens (norm 0,
    code of y = 0, decoded as exact zeros)."""
    for shared, kb, vb in ((True, 4, 4), (False, 4, 2)):
        got, want, _ = run_case(tq, orc, d=512, G=64, Hkv=1, B=1, L=1, chunks=[6], tails=[0], kb=kb, vb=vb,
                                shared=shared, end_to_end=False, seed=11, splits=1, scale=8.0, zero_every=7)
        _assert_close(got, want)


def test_tcgen05_d512_matches_mma_sync(tq, orc):
    """The tcgen05 and mma.sync kernels agree (same operand splits) and both
    meet the oracle, with two kv heads and separate K/V codecs."""
    cfg = dict(d=512, G=32, Hkv=2, B=1, L=1, chunks=[3], tails=[0], kb=3, vb=2, end_to_end=False, seed=9)
    a, want, _ = run_case(tq, orc, **cfg)
    b, _, _ = run_case(tq, orc, cuda_core_path=2, **cfg)
    _assert_close(a, want)
    _assert_close(b, want)
    assert np.max(np.abs(a - b)) <= 1e-4


@pytest.mark.parametrize("splits", [0, 1, 4])
def test_d512_dense_tail_tensor_cores(tq, orc, splits):
    """The tail on the tensor cores (16 heads a CTA, tokens in chunks of 32):
    ragged lengths over several chunks and splits, a ring that wraps, a batch
    with a one-token tail, a peaky softmax whose running maximum moves between
    chunks, two kv heads of 32 heads; the CUDA-core kernel gives the same."""
    cfg = dict(d=512, G=32, Hkv=2, B=3, L=1, chunks=[1, 2, 1], tails=[301, 33, 1], kb=3, vb=2, end_to_end=False,
               seed=21, scale=8.0, tail_cap=320, splits=splits)
    got, want, _ = run_case(tq, orc, **cfg)
    _assert_close(got, want)
    ref, _, _ = run_case(tq, orc, cuda_core_path=1, **cfg)
    assert np.max(np.abs(got - ref)) <= 1e-4


# soft cap 4 on logits of scale 6 (about N(0, 36)): most logits are capped.
# path: 0 automatic (tensor cores where they apply), 1 CUDA cores, 2 no tcgen05
SOFTCAP_CASES = [("tiny_gqa4_tail", 0), ("tiny_gqa4_tail", 1), ("qwen_like_gqa6", 0),
                 ("outliers_gqa4", 0), ("d256_mha_b1", 0), ("gqa3_odd_group", 0),
                 ("mqa_shared_d512", 0), ("mqa_shared_d512", 1), ("mqa_shared_d512", 2)]


@pytest.mark.parametrize("name,path", SOFTCAP_CASES)
def test_softcap(tq, orc, name, path):
    """Logit soft cap (arc PR #98, softcapping fix) on every kernel family:
    compressed and dense tokens, side lists, tcgen05 and mma.sync at d 512."""
    cfg = dict(CASES[name], scale=6.0, softcap=4.0, end_to_end=False, cuda_core_path=path)
    got, want, _ = run_case(tq, orc, **cfg)
    _assert_close(got, want)


def test_softcap_is_applied(tq, orc):
    """The capped GPU output is far from the uncapped oracle (the cap binds)."""
    cfg = dict(CASES["mqa_shared_d512"], scale=6.0, softcap=4.0, end_to_end=False)
    got, want, _ = run_case(tq, orc, oracle_softcap=0.0, **cfg)
    assert np.max(np.abs(got - want)) > 50 * TOL


def test_softcap_dense_layers(tq, orc):
    got, want, _ = run_case(tq, orc, d=128, G=6, Hkv=2, B=1, L=1, chunks=[0], tails=[600], kb=3, vb=2,
                            dense=True, scale=6.0, softcap=4.0)
    _assert_close(got, want)


def test_dense_boundary_layers(tq, orc):
    """bf16 layers: no records, the whole cache passed as the dense part."""
    got, want, _ = run_case(tq, orc, d=128, G=6, Hkv=2, B=1, L=2, chunks=[0], tails=[2048], kb=3, vb=2,
                            dense=True)
    _assert_close(got, want)


@pytest.mark.parametrize("path", PATHS)
def test_split_count_invariance(tq, orc, path):
    cfg = dict(d=128, G=4, Hkv=2, B=1, L=1, chunks=[12], tails=[100], kb=3, vb=2, end_to_end=False,
               cuda_core_path=(path == "cuda_core"))
    a, want, _ = run_case(tq, orc, splits=1, **cfg)
    b, _, _ = run_case(tq, orc, splits=40, **cfg)
    _assert_close(a, want)
    assert np.max(np.abs(a - b)) <= 1e-5


def test_many_splits_one_record_each(tq, orc):
    """70 records in 70 one-record splits (plus dense splits) against 4 splits:
    both agree with the oracle and with each other."""
    cfg = dict(d=64, G=2, Hkv=1, B=1, L=1, chunks=[70], tails=[20], kb=2, vb=2, end_to_end=False, seed=3)
    a, want, _ = run_case(tq, orc, splits=80, **cfg)
    b, _, _ = run_case(tq, orc, splits=4, **cfg)
    _assert_close(a, want)
    _assert_close(b, want)
    assert np.max(np.abs(a - b)) <= 1e-5


def test_empty_context_gives_zero(tq):
    import torch
    L, B, Hq, Hkv, d = 1, 2, 4, 2, 128
    q = torch.randn(L, B, Hq, d, device="cuda").to(torch.bfloat16)
    out = torch.full((L, B, Hq, d), float("nan"), device="cuda")
    kt = torch.zeros((L, B, Hkv, 16, d), dtype=torch.bfloat16, device="cuda")
    zero = torch.zeros((L, B), dtype=torch.int32, device="cuda")
    tq.decode_attn(q=q, out=out, scale=1.0, k_tail=kt, v_tail=kt, tail_start=zero, tail_len=zero, max_tail=16)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_single_token_returns_its_value(tq, orc):
    """One dense token: the output is that token's value (bf16 -> f32 exactly)."""
    got, want, _ = run_case(tq, orc, d=128, G=2, Hkv=1, B=1, L=1, chunks=[0], tails=[1], kb=3, vb=3,
                            end_to_end=False)
    _assert_close(got, want, tol=1e-6)
