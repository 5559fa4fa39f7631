"""Paged records and rollback on the GPU.

Paged records (arc PR #98 with the #94 head-dim generalisation: the paged
tq_attn kernel addresses the cache through a block table, byte offsets in 64
bits): a pool of blocks per layer, each holding one 128-token record per kv
head, and a [batch][table_stride] block table.  Attention over a shuffled
pool must equal attention over the same records laid out contiguously, on
every kernel route (bit for bit where the arithmetic order is fixed), and
eviction through the table must write the same bytes.

Rollback (arc PR #98, "What landed": truncation mapped onto both time bases;
a deep rollback dequantises): counters against the oracle's, the decoded
bf16 tail tokens against the oracle's bf16 rounding of its fp64 decode
(a one-step difference allowed only where the exact value lies within 1e-6
of a bf16 rounding midpoint, counted), records untouched, and attention over
the rolled-back cache against the oracle."""
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


def _cache(tq, *, L, B, Hkv, d, kb, vb, shared, T, R, seed):
    """Contiguous records [L, B, Hkv, R, bytes] of R full records per stream."""
    import torch
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = kc if shared else tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    n = L * B * Hkv
    kx = synth.gaussian_bf16((n, R * 128, d), seed, lognormal_sigma=0.3, outlier_frac=0.02 if T else 0.0)
    vx = kx if shared else synth.gaussian_bf16((n, R * 128, d), seed + 1)
    krec = torch.empty((L, B, Hkv, R, kc.record_bytes), dtype=torch.uint8, device="cuda")
    tq.tq_encode(kc, tl.to_bf16_tensor(kx, "cuda"), krec.view(n, R, -1))
    if shared:
        vrec = krec
    else:
        vrec = torch.empty((L, B, Hkv, R, vc.record_bytes), dtype=torch.uint8, device="cuda")
        tq.tq_encode(vc, tl.to_bf16_tensor(vx, "cuda"), vrec.view(n, R, -1))
    return kc, vc, krec, vrec


def _pool(rec, table, n_blocks):
    """The contiguous records [L, B, Hkv, R, bytes] scattered into a pool
    [L, n_blocks, Hkv, bytes] at block table[b][r] (other blocks hold junk)."""
    import torch
    L, B, Hkv, R, nb = rec.shape
    pool = torch.randint(0, 256, (L, n_blocks, Hkv, nb), dtype=torch.uint8, device=rec.device)
    for b in range(B):
        for r in range(R):
            pool[:, int(table[b, r])] = rec[:, b, :, r]
    return pool


ROUTES = [  # d, G, kb, vb, shared, T, cuda_core_path, route, exact
    (128, 6, 3, 2, False, 0.0, 0, "mma", True),
    (128, 4, 4, 3, False, 2.0, 0, "cuda_core_warp", False),
    (256, 4, 3, 2, False, 0.0, 0, "cuda_core", True),
    (512, 8, 4, 4, True, 0.0, 0, "mma512", True),
    (512, 64, 4, 4, True, 0.0, 0, "tcgen05", True),
]


@pytest.mark.parametrize("d,G,kb,vb,shared,T,path,route,exact", ROUTES)
def test_paged_attention_matches_contiguous(tq, orc, d, G, kb, vb, shared, T, path, route, exact):
    import torch
    L, B, R, tail = 2, 3, 4, 50
    Hkv = 1 if G == 64 else 2
    kc, vc, krec, vrec = _cache(tq, L=L, B=B, Hkv=Hkv, d=d, kb=kb, vb=vb, shared=shared, T=T, R=R, seed=71 + d)
    rng = np.random.default_rng(d + G)
    n_blocks = B * R + 5
    stride = R + 2                                    # table rows longer than the records in use
    perm = rng.permutation(n_blocks)
    table = np.full((B, stride), -7, np.int32)        # unused entries hold garbage
    table[:, :R] = perm[:B * R].reshape(B, R)
    tab = torch.from_numpy(table).cuda()
    kpool = _pool(krec, table, n_blocks)
    vpool = kpool if shared else _pool(vrec, table, n_blocks)
    kt = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, tail, d), 81), "cuda")
    vt = kt if shared else tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, tail, d), 82), "cuda")
    qb = synth.gaussian_bf16((L, B, G * Hkv, d), 83, scale=1 / math.sqrt(d))
    q = tl.to_bf16_tensor(qb, "cuda")
    nch = torch.tensor([[R, R - 1, 2]] * L, dtype=torch.int32, device="cuda")   # ragged record counts
    tlen = torch.full((L, B), tail, dtype=torch.int32, device="cuda")
    tstart = torch.full((L, B), 11, dtype=torch.int32, device="cuda")
    outs = []
    for paged in (False, True):
        out = torch.full((L, B, G * Hkv, d), float("nan"), dtype=torch.float32, device="cuda")
        kw = dict(q=q, out=out, scale=1.0, k_rec=kpool if paged else krec, v_rec=vpool if paged else vrec,
                  n_chunks=nch, max_chunks=R, k_tail=kt, v_tail=vt, tail_start=tstart, tail_len=tlen, max_tail=tail,
                  cuda_core_path=path, block_table=tab if paged else None)
        assert tq.tq_decode_attn_plan(tq.make_attn_args(**kw), kc, vc)["compressed_kernel"] == route
        tq.decode_attn(k_codec=kc, v_codec=vc, **kw)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert np.all(np.isfinite(outs[1]))
    if exact:
        np.testing.assert_array_equal(outs[1], outs[0])
    else:   # value corrections of outlier lists accumulate through shared-memory atomics
        assert float(np.max(np.abs(outs[1] - outs[0]))) <= 1e-6
    # one unit against the oracle
    okc, ovc = _ocodec(orc, kc), _ocodec(orc, vc)
    l, b, h = 1, 1, Hkv - 1
    kr, vr = krec[l, b, h].cpu().numpy(), vrec[l, b, h].cpu().numpy()
    slots = (11 + np.arange(tail)) % tail
    kd, vd = tl.bf16_tensor_bits(kt[l, b, h])[slots], tl.bf16_tensor_bits(vt[l, b, h])[slots]
    want = orc.unit_attention(qb[l, b, h * G:(h + 1) * G], okc, ovc, kr, vr, (R - 1) * 128, kd, vd, 1.0)
    assert float(np.max(np.abs(outs[1][l, b, h * G:(h + 1) * G] - want))) <= 2e-3


@pytest.mark.parametrize("d,kb,vb,shared,T", [(128, 4, 3, False, 2.0), (512, 4, 4, True, 0.0)])
def test_paged_eviction_matches_contiguous(tq, d, kb, vb, shared, T):
    import torch
    L, B, Hkv, R, cap = 2, 3, 2, 4, 272
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = kc if shared else tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    kt = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, cap, d), 91, outlier_frac=0.02 if T else 0.0), "cuda")
    vt = kt if shared else tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, cap, d), 92), "cuda")
    rng = np.random.default_rng(d)
    n_blocks = B * R + 3
    table = rng.permutation(n_blocks)[:B * R].reshape(B, R).astype(np.int32)
    tab = torch.from_numpy(table).cuda()
    res = []
    for paged in (False, True):
        shape = (L, n_blocks, Hkv) if paged else (L, B, Hkv, R)
        krec = torch.full(shape + (kc.record_bytes,), 0xCD, dtype=torch.uint8, device="cuda")
        vrec = krec if shared else torch.full(shape + (vc.record_bytes,), 0xCD, dtype=torch.uint8, device="cuda")
        nch = torch.tensor([[0, 1, 2]] * L, dtype=torch.int32, device="cuda")
        tstart = torch.tensor([[0, 200, 100]] * L, dtype=torch.int32, device="cuda")
        tlen = torch.tensor([[272, 272, 150]] * L, dtype=torch.int32, device="cuda")
        tq.tq_evict(kc, vc, k_rec=krec, v_rec=vrec, k_tail=kt, v_tail=vt, n_chunks=nch, tail_start=tstart,
                    tail_len=tlen, window=128, margin=16, t_q=1, max_evict=1, block_table=tab if paged else None)
        torch.cuda.synchronize()
        res.append((krec.cpu().numpy(), vrec.cpu().numpy(), nch.cpu().numpy(), tstart.cpu().numpy(),
                    tlen.cpu().numpy()))
    (k0, v0, *c0), (k1, v1, *c1) = res
    for a, bb in zip(c0, c1):
        np.testing.assert_array_equal(a, bb)
    np.testing.assert_array_equal(c1[0], [[1, 2, 2]] * L)     # batch 2 (150 tokens) evicts nothing
    for l in range(L):
        for b, r in ((0, 0), (1, 1)):
            np.testing.assert_array_equal(k1[l, table[b, r]], k0[l, b, :, r])
            np.testing.assert_array_equal(v1[l, table[b, r]], v0[l, b, :, r])
    # no other block of the pool was written
    written = {int(table[0, 0]), int(table[1, 1])}
    for blk in range(n_blocks):
        if blk not in written:
            assert np.all(k1[:, blk] == 0xCD)


CASES = [  # d, kb, vb, shared, T, scale, paged
    (64, 3, 2, False, 0.0, "norm", False),
    (128, 4, 3, False, 2.0, "norm", True),
    (256, 2, 2, False, 0.0, "least_squares", False),
    (512, 4, 4, True, 0.0, "norm", False),
]


@pytest.mark.parametrize("d,kb,vb,shared,T,scale,paged", CASES)
def test_rollback(tq, orc, d, kb, vb, shared, T, scale, paged):
    import torch
    L, B, Hkv, R, cap = 2, 3, 2, 4, 272
    kc, vc, krec, vrec = _cache(tq, L=L, B=B, Hkv=Hkv, d=d, kb=kb, vb=vb, shared=shared, T=T, R=R, seed=101 + d)
    if scale != "norm":   # re-encode with the scale variant
        kc = tq.with_scale(kc, scale)
        vc = kc if shared else tq.with_scale(vc, scale)
        n = L * B * Hkv
        kx = synth.gaussian_bf16((n, R * 128, d), 101 + d, lognormal_sigma=0.3, outlier_frac=0.02 if T else 0.0)
        vx = synth.gaussian_bf16((n, R * 128, d), 102 + d)
        tq.tq_encode(kc, tl.to_bf16_tensor(kx, "cuda"), krec.view(n, R, -1))
        tq.tq_encode(vc, tl.to_bf16_tensor(vx, "cuda"), vrec.view(n, R, -1))
    okc = _ocodec(orc, kc)
    okc = orc.Codec(d=okc.d, bits=okc.bits, T=okc.T, cap=okc.cap, scale=scale)
    ovc = okc if shared else orc.Codec(d=d, bits=vb, T=T, cap=okc.cap, scale=scale)
    kt = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, cap, d), 111), "cuda")
    vt = kt if shared else tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, cap, d), 112), "cuda")
    # per (layer, batch): n records in use, tail start/length, target length
    n_h = np.array([[4, 4, 3], [2, 4, 1]])
    s_h = np.array([[250, 0, 17], [100, 271, 5]])
    l_h = np.array([[200, 60, 130], [10, 271, 0]])
    totals = 128 * n_h + l_h
    new = np.array([[totals[0, 0], totals[0, 1] - 5, 2 * 128 + 127],   # no-op, within the tail, deep m = 127
                    [128, 10 ** 6, 77]])                                 # deep m = 0, clamp, deep into record 0
    table = None
    if paged:
        rng = np.random.default_rng(7)
        n_blocks = B * R + 2
        tabn = rng.permutation(n_blocks)[:B * R].reshape(B, R).astype(np.int32)
        table = torch.from_numpy(tabn).cuda()
        kr_dev = _pool(krec, tabn, n_blocks)
        vr_dev = kr_dev if shared else _pool(vrec, tabn, n_blocks)
    else:
        kr_dev, vr_dev = krec, vrec
    before = (kr_dev.clone(), vr_dev.clone())
    kt_host, vt_host = tl.bf16_tensor_bits(kt), tl.bf16_tensor_bits(vt)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    nch, tstart, tlen = i32(n_h), i32(s_h), i32(l_h)
    tq.tq_rollback(kc, vc, i32(new), k_rec=kr_dev, v_rec=vr_dev, k_tail=kt, v_tail=vt, n_chunks=nch,
                   tail_start=tstart, tail_len=tlen, block_table=table)
    torch.cuda.synchronize()
    assert torch.equal(kr_dev, before[0]) and torch.equal(vr_dev, before[1])     # records only read
    kr_h, vr_h = krec.cpu().numpy(), vrec.cpu().numpy()
    got_k, got_v = tl.bf16_tensor_bits(kt), tl.bf16_tensor_bits(vt)
    band = 0
    checked = 0
    for l in range(L):
        for b in range(B):
            tk, tv = kt_host[l, b].copy(), vt_host[l, b].copy()
            want = orc.rollback(tk, None if shared else tv, int(s_h[l, b]), int(l_h[l, b]), int(n_h[l, b]),
                                kr_h[l, b], None if shared else vr_h[l, b], okc, None if shared else ovc,
                                int(new[l, b]))
            assert (int(tstart[l, b]), int(tlen[l, b]), int(nch[l, b])) == want, (l, b)
            for gt, wt, rec, oc in ((got_k, tk, kr_h, okc), (got_v, tv, vr_h, ovc)):
                if shared and gt is got_v:
                    continue
                diff = gt[l, b] != wt
                if not diff.any():
                    continue
                # only the decoded slots may differ, by one bf16 step at a rounding midpoint
                m = want[1]
                assert want[0] == 0 and not diff[:, m:].any(), (l, b)
                x = np.stack([orc.decode_records(rec[l, b, h, want[2]:want[2] + 1], m, oc) for h in range(Hkv)])
                g16, w16 = gt[l, b][diff].astype(np.int64), wt[diff].astype(np.int64)
                assert np.all(np.abs(g16 - w16) == 1) and np.all(tl.bf16_midpoint_band(x[diff[:, :m]])), (l, b)
                band += int(diff.sum())
            checked += Hkv * want[1] * d
    assert band <= max(1, 1e-5 * checked)
    # attention over the rolled-back cache against the oracle
    G = 4
    qb = synth.gaussian_bf16((L, B, G * Hkv, d), 121, scale=1 / math.sqrt(d))
    out = torch.full((L, B, G * Hkv, d), float("nan"), dtype=torch.float32, device="cuda")
    tq.decode_attn(k_codec=kc, v_codec=vc, q=tl.to_bf16_tensor(qb, "cuda"), out=out, scale=1.0, k_rec=kr_dev,
                   v_rec=vr_dev, n_chunks=nch, max_chunks=R, k_tail=kt, v_tail=vt, tail_start=tstart, tail_len=tlen,
                   max_tail=cap, block_table=table)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for l in range(L):
        for b in range(B):
            n2, s2, l2 = int(nch[l, b]), int(tstart[l, b]), int(tlen[l, b])
            slots = (s2 + np.arange(l2)) % cap
            for h in range(Hkv):
                want = orc.unit_attention(qb[l, b, h * G:(h + 1) * G], okc, ovc, kr_h[l, b, h], vr_h[l, b, h],
                                          n2 * 128, got_k[l, b, h][slots], got_v[l, b, h][slots], 1.0)
                err = float(np.max(np.abs(got[l, b, h * G:(h + 1) * G] - want)))
                assert err <= 2e-3, (l, b, h, err)
