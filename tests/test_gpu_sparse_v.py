"""Sparse-V on the GPU (turboquant_plus commit log, "safer-asym + sparse-V
dequant"): the tensor-core decode kernel for head dims 64/128 skips the value
work of a warp's 32-token block when every logit of its CTA's heads there is
below the running maximum of the warp's earlier blocks plus ln(eps).  Checked
against the oracle applying the same rule on the kernel's schedule (taken from
tq_decode_attn_plan), against exact attention within the rule's bound, and
against the same call without skipping."""
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


@pytest.mark.parametrize("d,G,kb,vb,splits,T", [(128, 6, 3, 2, 2, 0.0), (64, 4, 4, 3, 3, 0.0), (128, 8, 4, 3, 0, 0.0),
                                               (128, 4, 4, 3, 2, 2.0)])
def test_sparse_v_matches_oracle_schedule(tq, orc, d, G, kb, vb, splits, T):
    import torch
    Hkv, R, tail, eps = 2, 12, 40, 2.0 ** -20
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    okc, ovc = orc.Codec(d=d, bits=kb, T=T), orc.Codec(d=d, bits=vb, T=T)
    ntok = R * 128
    qb = synth.gaussian_bf16((1, 1, G * Hkv, d), 5 + d, scale=2.0 / math.sqrt(d))
    q64 = synth.bf16_bits_to_f32(qb).astype(np.float64)[0, 0]
    k32 = synth.bf16_bits_to_f32(synth.gaussian_bf16((Hkv, ntok, d), 6 + d)).astype(np.float32)
    dev = "cuda"
    cnt = lambda v: torch.full((1, 1), v, dtype=torch.int32, device=dev)
    out = torch.empty((1, 1, G * Hkv, d), dtype=torch.float32, device=dev)
    # the schedule: records per split from the plan of this very call
    krec = torch.empty((1, 1, Hkv, R, kc.record_bytes), dtype=torch.uint8, device=dev)
    vrec = torch.empty((1, 1, Hkv, R, vc.record_bytes), dtype=torch.uint8, device=dev)
    kt = synth.gaussian_bf16((Hkv, tail, d), 7)
    vt = synth.gaussian_bf16((Hkv, tail, d), 8)
    kw = dict(q=tl.to_bf16_tensor(qb, dev), out=out, scale=1.0, k_rec=krec, v_rec=vrec, n_chunks=cnt(R),
              max_chunks=R, k_tail=tl.to_bf16_tensor(kt, dev)[None, None], v_tail=tl.to_bf16_tensor(vt, dev)[None, None],
              tail_start=cnt(0), tail_len=cnt(tail), max_tail=tail, splits=splits)
    plan = tq.tq_decode_attn_plan(tq.make_attn_args(**kw, sparse_v_eps=eps), kc, vc)
    assert plan["compressed_kernel"] == "mma"
    cps, gt, groups = plan["records_per_split"], plan["heads_per_cta"], plan["warps_per_cta"] // 4
    assert groups == (3 if T else 1)  # side lists: CTAs of three 4-warp groups
    # an attention sink (logit about 40 for every head of its kv head) opens
    # every (split, group, warp) sequence: later blocks fall far below it
    for h in range(Hkv):
        u = q64[h * G:(h + 1) * G].sum(0)
        sink = u * (40.0 / np.min(q64[h * G:(h + 1) * G] @ u))
        for s in range(0, R, cps):
            for g in range(min(groups, R - s, cps)):
                for w in range(4):
                    k32[h, 128 * (s + g) + 32 * w] = sink
    kx = synth.f32_to_bf16_bits(k32)
    vx = synth.gaussian_bf16((Hkv, ntok, d), 9 + d)
    tq.tq_encode(kc, tl.to_bf16_tensor(kx, dev), krec.view(Hkv, R, -1))
    tq.tq_encode(vc, tl.to_bf16_tensor(vx, dev), vrec.view(Hkv, R, -1))
    outs = {}
    for e in (0.0, eps):
        tq.decode_attn(k_codec=kc, v_codec=vc, sparse_v_eps=e, **kw)
        torch.cuda.synchronize()
        outs[e] = out.cpu().numpy()[0, 0].copy()
    kr, vr = krec.cpu().numpy()[0, 0], vrec.cpu().numpy()[0, 0]
    vmax = float(np.max(np.abs(orc.decode_records(vr[0], ntok, ovc))))
    total_skipped = 0
    for h in range(Hkv):
        qh = qb[0, 0, h * G:(h + 1) * G]
        want, skipped = orc.unit_attention_sparse_v(qh, okc, ovc, kr[h], vr[h], ntok, kt[h], vt[h], 1.0, eps,
                                                    cps, gt, groups=groups)
        exact = orc.unit_attention(qh, okc, ovc, kr[h], vr[h], ntok, kt[h], vt[h], 1.0)
        got = outs[eps][h * G:(h + 1) * G]
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - want))) <= 2e-3
        assert float(np.max(np.abs(got - exact))) <= 2e-3 + eps * skipped * vmax
        assert float(np.max(np.abs(got - outs[0.0][h * G:(h + 1) * G]))) <= 1e-5 + eps * skipped * vmax
        total_skipped += skipped
    # the sinks make most blocks skippable
    assert total_skipped >= 0.5 * Hkv * ntok * math.ceil(G / gt)


def test_sparse_v_other_routes_are_unsupported(tq):
    import torch
    dev = "cuda"
    for d, T, path in ((128, 2.0, 1), (256, 0.0, 0), (128, 0.0, 1)):
        kc = tq.tq_make_codebook(3, d, sign_seed=1, outlier_T=T)
        rec = torch.zeros((1, 1, 1, 2, kc.record_bytes), dtype=torch.uint8, device=dev)
        q = torch.zeros((1, 1, 4, d), dtype=torch.bfloat16, device=dev)
        out = torch.zeros((1, 1, 4, d), dtype=torch.float32, device=dev)
        n = torch.full((1, 1), 2, dtype=torch.int32, device=dev)
        a = tq.make_attn_args(q=q, out=out, scale=1.0, k_rec=rec, v_rec=rec, n_chunks=n, max_chunks=2,
                              cuda_core_path=path, sparse_v_eps=1e-3)
        with pytest.raises(tq.TqError) as e:
            tq.tq_decode_attn_plan(a, kc, kc)
        assert e.value.status == tq.TQ_ERR_UNSUPPORTED
        a.sparse_v_eps = 1.0                          # eps must lie in [0, 1)
        with pytest.raises(tq.TqError) as e:
            tq.tq_decode_attn_plan(a, kc, kc)
        assert e.value.status == tq.TQ_ERR_INVALID_ARG
