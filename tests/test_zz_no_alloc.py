"""tq_decode_attn_noalloc, the entry point for callers that cannot allocate
device memory when they run attention (memory reserved up front by a host
framework or pool, plugin enqueue steps that must not allocate, loops that
cannot take cudaMalloc's implicit synchronisation).  Its split-K workspace is
a fixed array inside the library, shared by every call and left holding the
previous call's contents, so each call here follows another of a different
shape: a d-128 call with many splits, a d-512 call on the tcgen05 route
(whose status word also lives in the array), a d-128 call with fewer splits,
and one with outlier side lists.  Each output must equal, bit for bit,
tq_decode_attn's with a fresh caller-allocated workspace (same plan, same
kernels; the outlier route, whose value corrections use shared-memory atomics,
within 1e-6) and match the oracle within the attention tolerance.  Collected
last on purpose: if it fails, a run stopping at the first failure has run
every other test."""
import ctypes
import math

import numpy as np
import pytest

import synth
import tq_testlib as tl

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _case(tq, dev, *, d, G, Hkv, kb, vb, shared, T, n_chunks, tail, seed):
    import torch
    L, B = 2, 2
    Hq = G * Hkv
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = kc if shared else tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    n = L * B * Hkv
    kx = synth.gaussian_bf16((n, n_chunks * 128, d), seed, outlier_frac=0.02 if T else 0.0, lognormal_sigma=0.3)
    vx = kx if shared else synth.gaussian_bf16((n, n_chunks * 128, d), seed + 1)
    krec = torch.empty((L, B, Hkv, n_chunks, kc.record_bytes), dtype=torch.uint8, device=dev)
    tq.tq_encode(kc, tl.to_bf16_tensor(kx, dev), krec.view(n, n_chunks, -1))
    if shared:
        vrec = krec
    else:
        vrec = torch.empty((L, B, Hkv, n_chunks, vc.record_bytes), dtype=torch.uint8, device=dev)
        tq.tq_encode(vc, tl.to_bf16_tensor(vx, dev), vrec.view(n, n_chunks, -1))
    kt = synth.gaussian_bf16((L, B, Hkv, tail, d), seed + 2)
    vt = kt if shared else synth.gaussian_bf16((L, B, Hkv, tail, d), seed + 3)
    q = synth.gaussian_bf16((L, B, Hq, d), seed + 4, scale=1 / math.sqrt(d))
    return dict(L=L, B=B, Hkv=Hkv, G=G, d=d, kc=kc, vc=vc, krec=krec, vrec=vrec, kt=kt, vt=vt, q=q,
                n_chunks=n_chunks, tail=tail)


def _run(tq, lib, c, dev, splits, noalloc):
    import torch
    L, B, G, Hkv, d = c["L"], c["B"], c["G"], c["Hkv"], c["d"]
    cnt = lambda v: torch.full((L, B), v, dtype=torch.int32, device=dev)
    out = torch.full((L, B, G * Hkv, d), float("nan"), dtype=torch.float32, device=dev)
    a = tq.make_attn_args(q=tl.to_bf16_tensor(c["q"], dev), out=out, scale=1.0, k_rec=c["krec"], v_rec=c["vrec"],
                          n_chunks=cnt(c["n_chunks"]), max_chunks=c["n_chunks"],
                          k_tail=tl.to_bf16_tensor(c["kt"], dev), v_tail=tl.to_bf16_tensor(c["vt"], dev),
                          tail_start=cnt(3), tail_len=cnt(c["tail"]), max_tail=c["tail"], splits=splits)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    kc, vc = ctypes.byref(c["kc"].c), ctypes.byref(c["vc"].c)
    if noalloc:
        st = lib.tq_decode_attn_noalloc(ctypes.byref(a), kc, vc, stream)
    else:
        need = lib.tq_decode_attn_workspace_size(ctypes.byref(a), kc, vc)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        st = lib.tq_decode_attn(ctypes.byref(a), kc, vc, ctypes.c_void_p(ws.data_ptr()), need, stream)
    assert st == tq.TQ_OK, tq.status_string(st)
    torch.cuda.synchronize()
    plan = tq.tq_decode_attn_plan(a, c["kc"], c["vc"])
    return out.cpu().numpy(), plan


def _oracle_check(orc, c, got):
    okc = orc.Codec(d=c["d"], bits=c["kc"].bits, T=float(c["kc"].c.outlier_T))
    ovc = orc.Codec(d=c["d"], bits=c["vc"].bits, T=float(c["vc"].c.outlier_T))
    kr, vr = c["krec"].cpu().numpy(), c["vrec"].cpu().numpy()
    G, tail = c["G"], c["tail"]
    for (l, b, h) in ((0, 0, 0), (c["L"] - 1, c["B"] - 1, c["Hkv"] - 1)):
        slots = (3 + np.arange(tail)) % tail
        want = orc.unit_attention(c["q"][l, b, h * G:(h + 1) * G], okc, ovc, kr[l, b, h], vr[l, b, h],
                                  c["n_chunks"] * 128, c["kt"][l, b, h][slots], c["vt"][l, b, h][slots], 1.0)
        err = float(np.max(np.abs(got[l, b, h * G:(h + 1) * G] - want)))
        assert err <= TOL, f"unit ({l},{b},{h}): max abs err {err} against the oracle"


def test_noalloc_matches_allocating_entry_point(orc):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rotated_lloyd_max_gb300 import build
    build.build()
    import rotated_lloyd_max_gb300 as tq
    lib = tq.load()
    dev = "cuda"
    d128 = _case(tq, dev, d=128, G=4, Hkv=2, kb=4, vb=3, shared=False, T=0.0, n_chunks=6, tail=60, seed=31)
    d512 = _case(tq, dev, d=512, G=32, Hkv=1, kb=4, vb=4, shared=True, T=0.0, n_chunks=3, tail=40, seed=41)
    outl = _case(tq, dev, d=128, G=4, Hkv=2, kb=4, vb=3, shared=False, T=2.0, n_chunks=5, tail=60, seed=51)
    calls = [(d128, 0, "mma", 0.0), (d512, 0, "tcgen05", 0.0), (d128, 2, "mma", 0.0), (outl, 0, None, 1e-6)]
    splits_seen = []
    for c, splits, kernel, tol in calls:
        got, plan = _run(tq, lib, c, dev, splits, noalloc=True)
        want, _ = _run(tq, lib, c, dev, splits, noalloc=False)
        if kernel is not None:
            assert plan["compressed_kernel"] == kernel
        splits_seen.append(plan["compressed_splits"])
        assert np.all(np.isfinite(got))
        if tol == 0.0:
            np.testing.assert_array_equal(got, want)
        else:
            assert float(np.max(np.abs(got - want))) <= tol
        _oracle_check(orc, c, got)
    assert splits_seen[2] < splits_seen[0], "the third call must use fewer splits than the first"


def test_noalloc_rejects_oversized_workspace():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rotated_lloyd_max_gb300 as tq
    lib = tq.load()
    L, B, Hq, d = 64, 64, 64, 512
    q = torch.zeros((1, 1, 8, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 1, 8, d), dtype=torch.float32, device="cuda")
    a = tq.make_attn_args(q=q, out=out, scale=1.0, k_tail=torch.zeros((1, 1, 1, 8, d), dtype=torch.bfloat16,
                                                                      device="cuda"),
                          v_tail=torch.zeros((1, 1, 1, 8, d), dtype=torch.bfloat16, device="cuda"),
                          tail_len=torch.zeros((1, 1), dtype=torch.int32, device="cuda"), max_tail=8)
    a.n_layers, a.batch, a.n_q_heads = L, B, Hq     # 64*64*64 rows x 512 floats > 8 MiB
    assert lib.tq_decode_attn_workspace_size(ctypes.byref(a), None, None) > tq.NOALLOC_WORKSPACE_BYTES
    st = lib.tq_decode_attn_noalloc(ctypes.byref(a), None, None,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == tq.TQ_ERR_WORKSPACE
