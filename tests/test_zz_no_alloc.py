"""tq_decode_attn_noalloc, the entry point for callers that cannot allocate
device memory when they run attention: it must give the same output as
tq_decode_attn with a caller-allocated workspace, on consecutive calls that
reuse its fixed library-owned workspace.  Collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest

import synth
import tq_testlib as tl

pytestmark = pytest.mark.gpu
TOL = 2e-3


def test_noalloc_matches_allocating_entry_point():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rotated_lloyd_max_gb300 import build
    build.build()
    import rotated_lloyd_max_gb300 as tq
    lib = tq.load()
    dev = "cuda"
    L, B, Hkv, G, d, n_chunks, tail = 2, 2, 2, 4, 128, 5, 60
    Hq = G * Hkv
    kc = tq.tq_make_codebook(4, d, sign_seed=1, outlier_T=2.0)
    vc = tq.tq_make_codebook(3, d, sign_seed=1, outlier_T=2.0)
    kx = tl.to_bf16_tensor(synth.gaussian_bf16((L * B * Hkv, n_chunks * 128, d), 31, outlier_frac=0.02), dev)
    vx = tl.to_bf16_tensor(synth.gaussian_bf16((L * B * Hkv, n_chunks * 128, d), 32), dev)
    krec = torch.empty((L, B, Hkv, n_chunks, kc.record_bytes), dtype=torch.uint8, device=dev)
    vrec = torch.empty((L, B, Hkv, n_chunks, vc.record_bytes), dtype=torch.uint8, device=dev)
    tq.tq_encode(kc, kx, krec.view(L * B * Hkv, n_chunks, -1))
    tq.tq_encode(vc, vx, vrec.view(L * B * Hkv, n_chunks, -1))
    kt = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, tail, d), 33), dev)
    vt = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hkv, tail, d), 34), dev)
    cnt = lambda v: torch.full((L, B), v, dtype=torch.int32, device=dev)
    for call in range(2):
        q = tl.to_bf16_tensor(synth.gaussian_bf16((L, B, Hq, d), 40 + call, scale=1 / math.sqrt(d)), dev)
        outs = []
        for noalloc in (False, True):
            out = torch.full((L, B, Hq, d), float("nan"), dtype=torch.float32, device=dev)
            a = tq.make_attn_args(q=q, out=out, scale=1.0, k_rec=krec, v_rec=vrec, n_chunks=cnt(n_chunks),
                                  max_chunks=n_chunks, k_tail=kt, v_tail=vt, tail_start=cnt(7),
                                  tail_len=cnt(tail), max_tail=tail)
            stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            if noalloc:
                st = lib.tq_decode_attn_noalloc(ctypes.byref(a), ctypes.byref(kc.c), ctypes.byref(vc.c), stream)
            else:
                need = lib.tq_decode_attn_workspace_size(ctypes.byref(a), ctypes.byref(kc.c), ctypes.byref(vc.c))
                ws = torch.empty(need, dtype=torch.uint8, device=dev)
                st = lib.tq_decode_attn(ctypes.byref(a), ctypes.byref(kc.c), ctypes.byref(vc.c),
                                        ctypes.c_void_p(ws.data_ptr()), need, stream)
            assert st == tq.TQ_OK, tq.status_string(st)
            torch.cuda.synchronize()
            outs.append(out.cpu().numpy())
        assert np.all(np.isfinite(outs[1]))
        assert np.max(np.abs(outs[0] - outs[1])) <= TOL


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
