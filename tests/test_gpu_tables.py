"""A caller-supplied centroid table end to end on the GPU ("v1.3 PPL on vLLM"
(PR #15), the calibrated Lloyd-Max commit: a sorted 2^b f32 table loaded in
place of the Gaussian one): tq_codec_set_centroids, then encode, decode and
decode attention on every attention route, each against the oracle run with
the same table."""
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


def _table(bits, d):
    """A symmetric ascending table that is not the Gaussian one: levels spread
    by a power law (wider outer levels), f32."""
    half = np.linspace(0.15, 2.2, 1 << (bits - 1)) ** 1.2
    return [float(v) for v in np.float32(np.concatenate([-half[::-1], half]) / math.sqrt(d))]


def _codecs(tq, orc, d, kb, vb, shared, T=0.0):
    kt, vt = _table(kb, d), _table(vb, d)
    kc = tq.tq_codec_set_centroids(tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T), kt)
    vc = kc if shared else tq.tq_codec_set_centroids(tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T), vt)
    cap = lambda c: int(c.c.outlier_cap) if T else 0
    okc = orc.Codec(d=d, bits=kb, T=T, cap=cap(kc), centroids=tuple(kt))
    ovc = okc if shared else orc.Codec(d=d, bits=vb, T=T, cap=cap(vc), centroids=tuple(vt))
    return kc, vc, okc, ovc


@pytest.mark.parametrize("d,bits", [(64, 2), (128, 3), (128, 4), (512, 4)])
def test_custom_table_codec(tq, orc, d, bits):
    import torch
    c, _, oc, _ = _codecs(tq, orc, d, bits, bits, True)
    n = 300
    x = synth.gaussian_bf16((n, d), 3000 + d + bits, lognormal_sigma=0.5)
    src = tl.to_bf16_tensor(x, "cuda")
    rec = torch.empty(((n + 127) // 128, c.record_bytes), dtype=torch.uint8, device="cuda")
    tq.tq_encode(c, src, rec)
    torch.cuda.synchronize()
    r = rec.cpu().numpy()
    codes, norms, _ = tl.unpack_records(r, n, d, bits)
    enc = orc.encode_vectors(x, oc, want_y=True)
    tl.check_codes(codes, enc, oc.tables()[1], d)
    tl.check_norms(norms, enc)
    dst = torch.empty((n, d), dtype=torch.float32, device="cuda")
    tq.tq_decode(c, rec, dst)
    err = float(np.max(np.abs(dst.cpu().numpy() - orc.decode_records(r, n, oc))))
    assert err <= 1e-5, f"decode max-abs {err}"


@pytest.mark.parametrize("d,G,kb,vb,shared,T,path,route", [
    (128, 6, 3, 2, False, 0.0, 0, "mma"),
    (128, 4, 4, 3, False, 2.0, 0, "cuda_core_warp"),
    (64, 4, 3, 3, False, 0.0, 1, "cuda_core_warp"),
    (512, 64, 4, 4, True, 0.0, 0, "tcgen05"),
    (512, 8, 4, 4, True, 0.0, 0, "mma512"),
])
def test_custom_table_attention(tq, orc, d, G, kb, vb, shared, T, path, route):
    import torch
    kc, vc, okc, ovc = _codecs(tq, orc, d, kb, vb, shared, T)
    Hkv, n_chunks, tail = 2 if G < 64 else 1, 3, 40
    ntok = n_chunks * 128
    dev = "cuda"
    kx = synth.gaussian_bf16((Hkv, ntok, d), 61 + d, lognormal_sigma=0.3, outlier_frac=0.02 if T else 0.0)
    vx = kx if shared else synth.gaussian_bf16((Hkv, ntok, d), 62 + d)
    kt = synth.gaussian_bf16((Hkv, tail, d), 63)
    vt = kt if shared else synth.gaussian_bf16((Hkv, tail, d), 64)
    q = synth.gaussian_bf16((1, 1, G * Hkv, d), 65, scale=1 / math.sqrt(d))
    krec = torch.empty((1, 1, Hkv, n_chunks, kc.record_bytes), dtype=torch.uint8, device=dev)
    tq.tq_encode(kc, tl.to_bf16_tensor(kx, dev), krec.view(Hkv, n_chunks, -1))
    if shared:
        vrec = krec
    else:
        vrec = torch.empty((1, 1, Hkv, n_chunks, vc.record_bytes), dtype=torch.uint8, device=dev)
        tq.tq_encode(vc, tl.to_bf16_tensor(vx, dev), vrec.view(Hkv, n_chunks, -1))
    out = torch.full((1, 1, G * Hkv, d), float("nan"), dtype=torch.float32, device=dev)
    cnt = lambda v: torch.full((1, 1), v, dtype=torch.int32, device=dev)
    kw = dict(q=tl.to_bf16_tensor(q, dev), out=out, scale=1.0, k_rec=krec, v_rec=vrec, n_chunks=cnt(n_chunks),
              max_chunks=n_chunks, k_tail=tl.to_bf16_tensor(kt, dev)[None, None],
              v_tail=tl.to_bf16_tensor(vt, dev)[None, None], tail_start=cnt(0), tail_len=cnt(tail), max_tail=tail,
              cuda_core_path=path)
    assert tq.tq_decode_attn_plan(tq.make_attn_args(**kw), kc, vc)["compressed_kernel"] == route
    tq.decode_attn(k_codec=kc, v_codec=vc, **kw)
    torch.cuda.synchronize()
    got = out.cpu().numpy()[0, 0]
    kr, vr = krec.cpu().numpy()[0, 0], vrec.cpu().numpy()[0, 0]
    for h in range(Hkv):
        want = orc.unit_attention(q[0, 0, h * G:(h + 1) * G], okc, ovc, kr[h], vr[h], ntok, kt[h], vt[h], 1.0)
        err = float(np.max(np.abs(got[h * G:(h + 1) * G] - want)))
        assert err <= 2e-3, f"kv head {h}: max abs err {err}"
