"""Parity at the workloads' full sizes, in the launch configuration the bench
times: inputs drawn on the device (the same recipes the bench uses), encoded
and attended by the library, then sampled (layer, batch, kv head) units and
records checked one by one against the oracle.  Sample sets always include
the last layer, batch, head and record (64-bit offsets past 4 GB)."""
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


def _bits(t):
    return tl.bf16_tensor_bits(t)


def _ocodec(orc, c):
    return orc.Codec(d=c.head_dim, bits=c.bits, seed=int(c.c.sign_seed), T=float(c.c.outlier_T),
                     cap=int(c.c.outlier_cap) if c.c.outlier_T else 0)


@pytest.fixture(autouse=True)
def _release_device_memory():
    """Each workload holds tens of GB: hand the cached blocks back after it."""
    yield
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()


class Cache:
    """A workload instantiated like the bench does (device-drawn inputs).
    With lean=True the bf16 inputs are drawn one layer at a time, encoded and
    dropped (only the records stay resident); sampled checks draw the layer
    again from its seed."""

    def __init__(self, tq, name, layers=None, batch=None, lean=False):
        import torch
        cfg = dict(synth.CONFIGS[name])
        self.cfg, self.tq = cfg, tq
        dev = "cuda"
        L = layers or cfg["L"]
        B = batch or cfg["B"]
        Hkv, Hq, d, ctx = cfg["Hkv"], cfg["Hq"], cfg["d"], cfg["ctx"]
        dense = [l for l in cfg.get("dense_layers", ()) if l < L]
        tail = cfg.get("tail", 0)
        n_rec = (ctx - tail) // 128
        self.L, self.B, self.Hkv, self.Hq, self.d, self.ctx, self.tail, self.n_rec = L, B, Hkv, Hq, d, ctx, tail, n_rec
        self.dense, self.shared = dense, cfg["shared_kv"]
        T = cfg["T"]
        self.kc = tq.tq_make_codebook(cfg["kb"], d, sign_seed=cfg["sign_seed"], outlier_T=T)
        self.vc = self.kc if self.shared else tq.tq_make_codebook(cfg["vb"], d, sign_seed=cfg["sign_seed"], outlier_T=T)
        seed = cfg["data_seed"]
        self.seed, self.lean = seed, lean
        bf = torch.bfloat16
        ntok = n_rec * 128
        self.ntok = ntok
        assert not (lean and (dense or tail)), "lean instantiation covers fully compressed caches"
        if lean:
            self.kx = self.vx = None
        else:
            self.kx = torch.empty((L, B, Hkv, ntok, d), dtype=bf, device=dev)
            self.vx = self.kx if self.shared else torch.empty_like(self.kx)
        self.q = torch.empty((L, B, Hq, d), dtype=bf, device=dev)
        tail_cap = max(tail, 1) if not dense else ctx
        self.kt = torch.zeros((L, B, Hkv, tail_cap, d), dtype=bf, device=dev)
        self.vt = self.kt if self.shared else torch.zeros_like(self.kt)
        for l in range(L):
            if not lean:
                self.layer_input(l, "k", out=self.kx[l])
                if not self.shared:
                    self.layer_input(l, "v", out=self.vx[l])
            synth.torch_gaussian_bf16(self.q[l].shape, synth.layer_seed(seed, l, 2), dev, scale=cfg["q_scale"],
                                      out=self.q[l])
            if tail:
                synth.torch_gaussian_bf16(self.kt[l, :, :, :tail].shape, synth.layer_seed(seed, l, 3), dev,
                                          out=self.kt[l, :, :, :tail], **synth.kv_recipe(cfg, "k"))
                if not self.shared:
                    synth.torch_gaussian_bf16(self.vt[l, :, :, :tail].shape, synth.layer_seed(seed, l, 4), dev,
                                              out=self.vt[l, :, :, :tail], **synth.kv_recipe(cfg, "v"))
        for l in dense:  # bf16 layers: the whole cache is the dense part
            self.kt[l].copy_(self.kx[l])
            self.vt[l].copy_(self.vx[l])
        u8, i32 = torch.uint8, torch.int32
        self.krec = torch.zeros((L, B, Hkv, n_rec, self.kc.record_bytes), dtype=u8, device=dev)
        self.vrec = self.krec if self.shared else torch.zeros((L, B, Hkv, n_rec, self.vc.record_bytes), dtype=u8,
                                                              device=dev)
        comp = [l for l in range(L) if l not in dense]
        n = B * Hkv
        for l in comp:
            kx = self.layer_input(l, "k") if lean else self.kx[l]
            tq.tq_encode(self.kc, kx.view(n, ntok, d), self.krec[l].view(n, n_rec, -1))
            del kx
            if not self.shared:
                vx = self.layer_input(l, "v") if lean else self.vx[l]
                tq.tq_encode(self.vc, vx.view(n, ntok, d), self.vrec[l].view(n, n_rec, -1))
                del vx
        self.n_chunks = torch.tensor([[0 if l in dense else n_rec] * B for l in range(L)], dtype=i32, device=dev)
        self.tail_len = torch.tensor([[ctx if l in dense else tail] * B for l in range(L)], dtype=i32, device=dev)
        self.out = torch.full((L, B, Hq, d), float("nan"), dtype=torch.float32, device=dev)
        kw = dict(q=self.q, out=self.out, scale=1.0, k_rec=self.krec, v_rec=self.vrec, n_chunks=self.n_chunks,
                  max_chunks=n_rec)
        if tail or dense:
            kw.update(k_tail=self.kt, v_tail=self.vt, tail_len=self.tail_len, max_tail=int(self.tail_len.max()))
        tq.decode_attn(k_codec=self.kc, v_codec=self.vc, **kw)
        torch.cuda.synchronize()

    def layer_input(self, l, stream, out=None):
        """Layer l's packed-region K ("k") or V ("v") draw, bf16 [B, Hkv, ntok, d]."""
        import torch
        shape = (self.B, self.Hkv, self.ntok, self.d)
        if out is None:
            out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        return synth.torch_gaussian_bf16(shape, synth.layer_seed(self.seed, l, 0 if stream == "k" else 1), "cuda",
                                         out=out, **synth.kv_recipe(self.cfg, stream))

    def check_unit(self, orc, l, b, h, n_rec_checked=3, tally=None):
        cfg, d, G = self.cfg, self.d, self.Hq // self.Hkv
        okc, ovc = _ocodec(orc, self.kc), _ocodec(orc, self.vc)
        q = _bits(self.q[l, b, h * G:(h + 1) * G])
        if l in self.dense:
            kd, vd = _bits(self.kt[l, b, h]), _bits(self.vt[l, b, h])
            want = orc.unit_attention(q, None, None, None, None, 0, kd, vd, 1.0)
        else:
            kr = self.krec[l, b, h].cpu().numpy()
            vr = self.vrec[l, b, h].cpu().numpy()
            kd = _bits(self.kt[l, b, h, :self.tail]) if self.tail else None
            vd = _bits(self.vt[l, b, h, :self.tail]) if self.tail else None
            want = orc.unit_attention(q, okc, ovc, kr, vr, self.n_rec * 128, kd, vd, 1.0)
            # records: first, last and one in the middle, against the oracle's encode
            if self.lean:
                kx = self.layer_input(l, "k")[b, h]
                srcs = (kx, kx if self.shared else self.layer_input(l, "v")[b, h])
            else:
                srcs = (self.kx[l, b, h], self.vx[l, b, h])
            for r in sorted({0, self.n_rec // 2, self.n_rec - 1})[:n_rec_checked]:
                for oc, rec, src in ((okc, kr, srcs[0]), (ovc, vr, srcs[1])):
                    x = _bits(src[r * 128:(r + 1) * 128])
                    codes, norms, outs = tl.unpack_records(rec[r], 128, d, oc.bits, oc.has_outliers,
                                                           oc.outlier_cap if oc.has_outliers else 0)
                    enc = orc.encode_vectors(x, oc, want_y=True)
                    tally.add(codes, enc, orc.codebook_f32(oc.bits, d)[1], d)
                    tl.check_norms(norms, enc)
                    if oc.has_outliers:
                        tally.add_outliers(outs, enc, d, oc.T)
        got = self.out[l, b, h * G:(h + 1) * G].cpu().numpy()
        assert np.all(np.isfinite(got))
        err = float(np.max(np.abs(got - want)))
        assert err <= TOL, f"unit ({l},{b},{h}): max abs err {err}"
        return err


def test_qwen2_cache_every_unit(tq, orc):
    """28 layers (6 bf16), all 56 (layer, kv head) units checked."""
    c = Cache(tq, "qwen2_1p5b_ctx2048")
    tally = tl.MismatchTally()
    for l in range(c.L):
        for h in range(c.Hkv):
            c.check_unit(orc, l, 0, h, n_rec_checked=3, tally=tally)
    tally.check()


def test_v4flash_mqa_full_context(tq, orc):
    """43 layers, 65,280 packed + 256 tail tokens, 64 query heads on one kv head."""
    c = Cache(tq, "v4flash_mqa_ctx65536")
    tally = tl.MismatchTally()
    for l in (0, 21, 42):
        c.check_unit(orc, l, 0, 0, tally=tally)
    tally.check()


def test_batched_outliers(tq, orc):
    """Batch 32 x 8 kv heads x 32,768 tokens with outlier side lists, all 32
    layers (55 GB of records) in one tq_decode_attn call, as the bench runs it;
    the bf16 inputs are drawn layer by layer and dropped after encoding."""
    c = Cache(tq, "batched_b32_ctx32768", lean=True)
    assert c.L == 32
    tally = tl.MismatchTally()
    for (l, b, h) in ((0, 0, 0), (31, 31, 7), (17, 17, 5), (6, 6, 2)):
        c.check_unit(orc, l, b, h, n_rec_checked=3, tally=tally)
    tally.check()


def test_long_context(tq, orc):
    """Batch 4 x 8 kv heads x 262,144 tokens (1,024 dense), 8 layers; records of
    a layer exceed 2 GB, so the last units exercise 64-bit offsets."""
    c = Cache(tq, "longctx_b4_ctx262144")
    tally = tl.MismatchTally()
    for (l, b, h) in ((0, 0, 0), (7, 3, 7), (4, 2, 3)):
        c.check_unit(orc, l, b, h, n_rec_checked=3, tally=tally)
    tally.check()


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_encode_sweep_full_size(tq, orc, d):
    """2^24 N(0,1) vectors per head dim and bit width, encoded in one call;
    a spread sample of records (first, last, and random) checked."""
    import torch
    n = 1 << 24
    x = synth.torch_gaussian_bf16((n, d), synth.layer_seed(0, d, 0), "cuda")
    rng = np.random.default_rng(d)
    nrec = n // 128
    picks = sorted({0, nrec - 1, *rng.integers(0, nrec, 6).tolist()})
    tally = tl.MismatchTally()
    for bits in (2, 3, 4):
        c = tq.tq_make_codebook(bits, d, sign_seed=1)
        rec = torch.empty((nrec, c.record_bytes), dtype=torch.uint8, device="cuda")
        tq.tq_encode(c, x, rec)
        torch.cuda.synchronize()
        oc = _ocodec(orc, c)
        for r in picks:
            xs = _bits(x[r * 128:(r + 1) * 128])
            codes, norms, _ = tl.unpack_records(rec[r].cpu().numpy(), 128, d, bits)
            enc = orc.encode_vectors(xs, oc, want_y=True)
            tally.add(codes, enc, orc.codebook_f32(bits, d)[1], d)
            tl.check_norms(norms, enc)
        del rec
    tally.check()
    del x
    torch.cuda.empty_cache()
