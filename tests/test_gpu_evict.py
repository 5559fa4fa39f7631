"""GPU parity of chunked eviction (tq_evict) against the oracle's eviction
bookkeeping and encode: device-side decisions, record contents, counters, the
append-only property and the tail staying exact."""
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


@pytest.mark.parametrize("shared,d,kb,vb,T", [(False, 128, 4, 3, 0.0), (True, 512, 4, 4, 0.0),
                                              (False, 64, 3, 2, 2.0)])
def test_chunked_eviction(tq, orc, shared, d, kb, vb, T):
    import torch
    L, B, Hkv, cap, rec_cap = 2, 2, 2, 544, 6
    window, margin, t_q = 128, 16, 1
    kc = tq.tq_make_codebook(kb, d, sign_seed=1, outlier_T=T)
    vc = kc if shared else tq.tq_make_codebook(vb, d, sign_seed=1, outlier_T=T)
    okc, ovc = _ocodec(orc, kc), _ocodec(orc, vc)
    ntot = 900
    toks_k = synth.gaussian_bf16((L, B, Hkv, ntot, d), 21, lognormal_sigma=0.3)
    toks_v = toks_k if shared else synth.gaussian_bf16((L, B, Hkv, ntot, d), 22)
    dev = "cuda"
    ktail = torch.zeros((L, B, Hkv, cap, d), dtype=torch.bfloat16, device=dev)
    vtail = ktail if shared else torch.zeros_like(ktail)
    krec = torch.full((L, B, Hkv, rec_cap, kc.record_bytes), 0xCD, dtype=torch.uint8, device=dev)
    vrec = krec if shared else torch.full((L, B, Hkv, rec_cap, vc.record_bytes), 0xCD, dtype=torch.uint8,
                                          device=dev)
    n_chunks = torch.zeros((L, B), dtype=torch.int32, device=dev)
    tstart = torch.zeros((L, B), dtype=torch.int32, device=dev)
    tlen = torch.zeros((L, B), dtype=torch.int32, device=dev)
    # batch 1 starts later than batch 0 so their evictions fall at different steps
    offset = [0, 100]
    host = dict(start=np.zeros((L, B), int), length=np.zeros((L, B), int), n=np.zeros((L, B), int))
    snapshots = []
    step_sizes = [271, 1, 60, 70, 129, 1, 256, 100]   # includes a two-chunk step (max_evict = 2)
    pos = np.zeros(B, int)
    for st in step_sizes:
        for b in range(B):
            n_new = max(0, min(st - (offset[b] if pos[b] == 0 else 0), ntot - pos[b]))
            for l in range(L):
                s0, ln = host["start"][l, b], host["length"][l, b]
                slots = (s0 + ln + np.arange(n_new)) % cap
                sl = torch.from_numpy(slots).to(dev)
                ktail[l, b][:, sl] = tl.to_bf16_tensor(toks_k[l, b, :, pos[b]:pos[b] + n_new], dev)
                if not shared:
                    vtail[l, b][:, sl] = tl.to_bf16_tensor(toks_v[l, b, :, pos[b]:pos[b] + n_new], dev)
                host["length"][l, b] += n_new
            pos[b] += n_new
        tlen.copy_(torch.from_numpy(host["length"].astype(np.int32)))
        tq.tq_evict(kc, vc, k_rec=krec, v_rec=vrec, k_tail=ktail, v_tail=vtail, n_chunks=n_chunks,
                    tail_start=tstart, tail_len=tlen, window=window, margin=margin, t_q=t_q, max_evict=2)
        torch.cuda.synchronize()
        for l in range(L):
            for b in range(B):
                k = orc.chunks_to_evict(int(host["length"][l, b]), window, t_q, margin)
                k = min(k, 2)
                host["n"][l, b] += k
                host["start"][l, b] = (host["start"][l, b] + 128 * k) % cap
                host["length"][l, b] -= 128 * k
        np.testing.assert_array_equal(n_chunks.cpu().numpy(), host["n"])
        np.testing.assert_array_equal(tstart.cpu().numpy(), host["start"])
        np.testing.assert_array_equal(tlen.cpu().numpy(), host["length"])
        snapshots.append((krec.cpu().numpy().copy(), host["n"].copy()))
    assert host["n"].min() >= 3
    # append-only: a record, once written, never changes
    for (a, na), (b_, _) in zip(snapshots, snapshots[1:]):
        for l in range(L):
            for b in range(B):
                np.testing.assert_array_equal(a[l, b, :, :na[l, b]], b_[l, b, :, :na[l, b]])
    # record r of (l, b, h) holds tokens [128 r, 128 r + 128) of that stream
    kr, vr = krec.cpu().numpy(), vrec.cpu().numpy()
    tally = tl.MismatchTally()
    for l in range(L):
        for b in range(B):
            n = host["n"][l, b]
            assert np.all(kr[l, b, :, n:] == 0xCD)
            for h in range(Hkv):
                for stream, oc, rec, src in (("k", okc, kr, toks_k), ("v", ovc, vr, toks_v)):
                    if shared and stream == "v":
                        continue
                    x = src[l, b, h, :128 * n]
                    codes, norms, outs = tl.unpack_records(rec[l, b, h], 128 * n, d, oc.bits, oc.has_outliers,
                                                           oc.outlier_cap if oc.has_outliers else 0)
                    enc = orc.encode_vectors(x, oc, want_y=True)
                    tally.add(codes, enc, orc.codebook_f32(oc.bits, d)[1], d)
                    tl.check_norms(norms, enc)
                    if oc.has_outliers:
                        tally.add_outliers(outs, enc, d, oc.T)
            # the tail still holds exactly the newest tokens
            slots = (host["start"][l, b] + np.arange(host["length"][l, b])) % cap
            tail = tl.bf16_tensor_bits(ktail[l, b][:, torch.from_numpy(slots).to(dev)])
            first = 128 * host["n"][l, b]
            np.testing.assert_array_equal(tail, toks_k[l, b, :, first:first + host["length"][l, b]])
    tally.check()


def test_v4flash_cache_grown_by_eviction(tq, orc):
    """The V4-Flash-like cache (43 layers, one kv head, head dim 512, keys and
    values sharing 4-bit records) grown to its full 65,536-token context through
    tq_evict alone: tokens enter the 272-slot ring 128 at a time (the first
    step 272) and every call evicts the chunk that reached the bound
    window 128 + max(t_q - 1, margin 16) + 128.  Afterwards 510 records and a
    256-token tail per layer; sampled records against the oracle's encode, the
    counters against the oracle's eviction arithmetic, and the decode
    attention over the grown cache against the oracle for three layers."""
    import torch
    cfg = synth.CONFIGS["v4flash_mqa_ctx65536"]
    L, d, ctx, G = cfg["L"], cfg["d"], cfg["ctx"], cfg["Hq"]
    window, margin, t_q = cfg["window"], cfg["margin"], cfg["t_q"]
    cap = window + max(t_q - 1, margin) + 128
    rec_cap = ctx // 128
    kc = tq.tq_make_codebook(cfg["kb"], d, sign_seed=cfg["sign_seed"])
    okc = _ocodec(orc, kc)
    dev = "cuda"
    x = torch.empty((L, ctx, d), dtype=torch.bfloat16, device=dev)
    for l in range(L):
        synth.torch_gaussian_bf16((ctx, d), synth.layer_seed(cfg["data_seed"], l, 0), dev, out=x[l],
                                  **synth.kv_recipe(cfg, "k"))
    tail = torch.zeros((L, 1, 1, cap, d), dtype=torch.bfloat16, device=dev)
    rec = torch.full((L, 1, 1, rec_cap, kc.record_bytes), 0xCD, dtype=torch.uint8, device=dev)
    n_chunks = torch.zeros((L, 1), dtype=torch.int32, device=dev)
    tstart = torch.zeros((L, 1), dtype=torch.int32, device=dev)
    tlen = torch.zeros((L, 1), dtype=torch.int32, device=dev)
    h_start, h_len, h_n, pos = 0, 0, 0, 0
    while pos < ctx:
        n_new = min(cap - h_len, ctx - pos)
        slots = torch.from_numpy((h_start + h_len + np.arange(n_new)) % cap).to(dev)
        tail[:, 0, 0, slots] = x[:, pos:pos + n_new]
        pos += n_new
        h_len += n_new
        tlen += n_new                         # the host appends; eviction runs on the device
        tq.tq_evict(kc, kc, k_rec=rec, v_rec=rec, k_tail=tail, v_tail=tail, n_chunks=n_chunks,
                    tail_start=tstart, tail_len=tlen, window=window, margin=margin, t_q=t_q, max_evict=1)
        k = min(orc.chunks_to_evict(h_len, window, t_q, margin), 1)
        h_n += k
        h_start = (h_start + 128 * k) % cap
        h_len -= 128 * k
    torch.cuda.synchronize()
    assert (h_n, h_len) == (510, 256)
    assert torch.all(n_chunks == h_n) and torch.all(tstart == h_start) and torch.all(tlen == h_len)
    assert torch.all(rec[:, :, :, h_n:] == 0xCD)     # nothing past the last evicted record
    tally = tl.MismatchTally()
    rng = np.random.default_rng(43)
    for l in (0, 21, 42):
        rl = rec[l, 0, 0].cpu().numpy()
        for r in sorted({0, 1, h_n - 1, *rng.integers(0, h_n, 3).tolist()}):
            xs = tl.bf16_tensor_bits(x[l, r * 128:(r + 1) * 128])
            codes, norms, _ = tl.unpack_records(rl[r], 128, d, okc.bits)
            enc = orc.encode_vectors(xs, okc, want_y=True)
            tally.add(codes, enc, orc.codebook_f32(okc.bits, d)[1], d)
            tl.check_norms(norms, enc)
    tally.check()
    # decode attention over the grown cache (tcgen05 records + the ring tail)
    q = torch.empty((L, 1, G, d), dtype=torch.bfloat16, device=dev)
    for l in range(L):
        synth.torch_gaussian_bf16((1, G, d), synth.layer_seed(cfg["data_seed"], l, 2), dev, scale=cfg["q_scale"],
                                  out=q[l])
    out = torch.full((L, 1, G, d), float("nan"), dtype=torch.float32, device=dev)
    tq.decode_attn(k_codec=kc, v_codec=kc, q=q, out=out, scale=1.0, k_rec=rec, v_rec=rec, n_chunks=n_chunks,
                   max_chunks=rec_cap, k_tail=tail, v_tail=tail, tail_start=tstart, tail_len=tlen, max_tail=cap)
    torch.cuda.synchronize()
    slots = (h_start + np.arange(h_len)) % cap
    for l in (0, 21, 42):
        kd = tl.bf16_tensor_bits(tail[l, 0, 0])[slots]
        np.testing.assert_array_equal(kd, tl.bf16_tensor_bits(x[l, 128 * h_n:]))
        rl = rec[l, 0, 0].cpu().numpy()
        want = orc.unit_attention(tl.bf16_tensor_bits(q[l, 0]), okc, okc, rl, rl, 128 * h_n, kd, kd, 1.0)
        got = out[l, 0].cpu().numpy()
        err = float(np.max(np.abs(got - want)))
        assert np.all(np.isfinite(got)) and err <= 2e-3, f"layer {l}: attention max abs err {err}"
