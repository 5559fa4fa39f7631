#!/usr/bin/env python
"""Benchmark of the rotated Lloyd-Max KV-cache path on GB300.

Default workload: the batched decode cache (32 layers, batch 32, 8 KV heads,
32 query heads, head_dim 128, ctx 32,768; K 4 bits, V 3 bits, outlier side
lists at T = 2 on both), the largest configuration that fits one GPU (about
193 GB resident).  One step = three phases, each replayed from a CUDA graph
and timed with CUDA events on the launching stream, with L2 flushed (a 256 MiB
write) before each phase outside its events:
  encode     tq_encode of the whole compressed cache (K and V),
  eviction   one tq_evict call moving one 128-token chunk per (layer, batch,
             kv head) from its dense ring into a record,
  attention  one decode step of every layer in one tq_decode_attn call.
Inputs are synthetic, generated on the device from fixed seeds, resident in
HBM before timing.

value = algorithmic HBM bytes of the step (bytes each kernel must read and
write by the record layout) / device time, in GB/s.  Also reported: encode
Mvec/s, eviction Mvec/s, decode-attention KV GB/s and tok/s, the roofline of
every phase against the measured HBM copy bandwidth (attention above the
ridge point against the measured bf16 tensor peak) with the dominant phase as
`roofline`, the oracle (CPU) timed on a bounded sample, and an end-to-end
figure with host buffers copied in and out.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload batched_b32_ctx32768|qwen2_1p5b_ctx2048|v4flash_mqa_ctx65536
                              |longctx_b4_ctx262144|codec_roundtrip_4096x128_b3|encode_sweep_16M]
                  [--splits N] [--layers L] [--batch B]
Under torchrun (N > 1) every rank runs an independent replica of the workload
(the path has no cross-GPU exchange); value = total bytes of all ranks / max
rank time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 20 for the large caches, 5000 for the Qwen2 cache)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="batched_b32_ctx32768",
                    choices=["batched_b32_ctx32768", "qwen2_1p5b_ctx2048", "v4flash_mqa_ctx65536",
                             "longctx_b4_ctx262144", "codec_roundtrip_4096x128_b3", "encode_sweep_16M"])
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="cache workloads: instantiate only the first L layers (small profiling cases)")
    ap.add_argument("--batch", type=int, default=None, help="cache workloads: instantiate batch B")
    ap.add_argument("--splits", type=int, default=0,
                    help="cache workloads: splits per (layer, batch, kv head) of tq_decode_attn (0 = its planner)")
    ap.add_argument("--sparse-v", type=float, default=0.0,
                    help="cache workloads on the d-64/128 tensor-core route: sparse-V threshold eps (0 = off); "
                         "the attention phase is also timed without it")
    ap.add_argument("--sinks", action="store_true",
                    help="cache workloads: plant an attention-sink key (logit about 40 for every head of its kv "
                         "head) at the first token of every 32-token block the decode kernel's warps open a "
                         "split with")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("TQ_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.proc = None
        self.lines = []
        self.idx = device_index
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms",
                     "200", "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                    text=True)
            except (OSError, ValueError):
                self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
# Eviction bound of the cache workloads: window + max(t_q - 1, margin) + 128
# ("feat(v4): TurboQuant KV storage for DeepSeek-V4", "Eviction is chunked, on
# purpose"); the V4-Flash-like config states window 128, the others take the
# same values.
EVICT_WINDOW, EVICT_MARGIN, EVICT_TQ = 128, 16, 1

# DRAM bytes (read + write) per step of a phase, from dram__bytes_read.sum +
# dram__bytes_write.sum of a one-kernel ncu capture, keyed by the SHA-256
# (first 16 hex digits) of the phase's kernel sources at capture time; a
# phase whose sources have changed since reports null.  Captures of a reduced
# layer count are scaled to the full workload by layers (the phase's traffic
# is a sum over layers).
# Captured at commit 54b393f (profiles/phase_traffic.md): small cases
# (batched --layers 2, V4-Flash-like --layers 8, long context --layers 1,
# Qwen2-shaped in full), mean over the captured steps, scaled by layers.
_T = {"tq_encode": "cf493c19144d20f9", "tq_evict": "cb3934c670ca7e8f", "tq_decode_attn": "4990717f4be6d7ec"}
MEASURED_TRAFFIC: dict = {
    ("batched_b32_ctx32768", "tq_encode"): {"bytes": 181_461_894_758, "sources": _T["tq_encode"]},
    ("batched_b32_ctx32768", "tq_evict"): {"bytes": 538_411_827, "sources": _T["tq_evict"]},
    ("batched_b32_ctx32768", "tq_decode_attn"): {"bytes": 45_096_975_565, "sources": _T["tq_decode_attn"]},
    ("v4flash_mqa_ctx65536", "tq_encode"): {"bytes": 3_494_490_632, "sources": _T["tq_encode"]},
    ("v4flash_mqa_ctx65536", "tq_evict"): {"bytes": 5_780_232, "sources": _T["tq_evict"]},
    ("v4flash_mqa_ctx65536", "tq_decode_attn"): {"bytes": 866_984_370, "sources": _T["tq_decode_attn"]},
    ("longctx_b4_ctx262144", "tq_encode"): {"bytes": 39_890_091_622, "sources": _T["tq_encode"]},
    ("longctx_b4_ctx262144", "tq_evict"): {"bytes": 17_132_339, "sources": _T["tq_evict"]},
    ("longctx_b4_ctx262144", "tq_decode_attn"): {"bytes": 6_100_180_992, "sources": _T["tq_decode_attn"]},
    ("qwen2_1p5b_ctx2048", "tq_encode"): {"bytes": 46_205_952, "sources": _T["tq_encode"]},
    ("qwen2_1p5b_ctx2048", "tq_evict"): {"bytes": 2_927_667, "sources": _T["tq_evict"]},
    ("qwen2_1p5b_ctx2048", "tq_decode_attn"): {"bytes": 22_128_998, "sources": _T["tq_decode_attn"]},
}

PHASE_SOURCES = {
    "tq_encode": ["encode_mma.cuh", "encode_mma.cu", "encode_mma_d64.cu", "encode_mma_d256.cu", "encode_mma_d512.cu",
                  "tq_common.cuh", "tq_params.h", "abi.cu"],
    "tq_evict": ["evict.cu", "encode_core.cuh", "tq_common.cuh", "tq_params.h", "abi.cu"],
    "tq_decode_attn": ["abi.cu", "merge.cu", "umma.cuh", "tq_common.cuh", "tq_params.h",
                       "attn.cuh", "attn_rec.cuh", "attn_mma.cuh", "attn_mma512.cuh", "attn_umma512.cuh",
                       "attn_dense512.cuh"],
}


def phase_sources_sha(phase: str) -> str:
    """SHA-256 (16 hex digits) of the library sources a phase's kernels are built from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rotated_lloyd_max_gb300", "csrc")
    for name in PHASE_SOURCES[phase]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, phase: str):
    e = MEASURED_TRAFFIC.get((workload, phase))
    if e is None or e["sources"] != phase_sources_sha(phase):
        return None
    return e["bytes"]


def peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, "measured" | "fallback")."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def used_record_bytes(torch, rec, codec, d: int) -> int:
    """Algorithmic bytes of a record array [..., record_bytes]: codes and norms
    of every record, plus the outlier counts and the entries actually stored."""
    base = 128 * (d * codec.bits // 8) + 512
    flat = rec.reshape(-1, codec.record_bytes)
    n = flat.shape[0]
    if not codec.c.outlier_T:
        return n * base
    entries = int(flat[:, base:base + 128].to(torch.int64).sum().item())
    return n * (base + 128) + 4 * entries


class EvictPhase:
    """One tq_evict call that evicts one 128-token chunk for every compressed
    (layer, batch, kv head) of a cache: each stream gets a 272-slot bf16 ring
    (window 128 + margin 16 + one chunk) whose oldest 128 slots hold the
    tokens of the stream's last record and whose other 144 slots hold newer
    tokens; its counters (n_chunks = records - 1, start 0, length 272) are
    reset from device templates before every call, so each call re-evicts
    that record with the same tokens, as a decode step that fills a chunk
    does."""

    def __init__(self, wl, layers: slice, next_k, next_v):
        torch = wl.torch
        self.wl, self.tq, self.torch = wl, wl.tq, torch
        cap = EVICT_WINDOW + max(EVICT_TQ - 1, EVICT_MARGIN) + 128
        self.cap = cap
        kx = wl.kx[layers]
        Lc, B, Hkv = kx.shape[:3]
        d, nt = wl.d, wl.n_rec * 128
        self.krec, self.vrec = wl.krec[layers], wl.vrec[layers]
        self.kt = torch.cat([kx[:, :, :, nt - 128:nt], next_k], dim=3).contiguous()
        assert self.kt.shape[3] == cap
        if wl.shared:
            self.vt = self.kt
        else:
            self.vt = torch.cat([wl.vx[layers][:, :, :, nt - 128:nt], next_v], dim=3).contiguous()
        i32 = torch.int32
        dev = kx.device
        self.tmpl = [torch.full((Lc, B), v, dtype=i32, device=dev) for v in (wl.n_rec - 1, 0, cap)]
        self.n_chunks, self.tail_start, self.tail_len = [t.clone() for t in self.tmpl]
        self.streams = 1 if wl.shared else 2
        self.launches = self.streams + 1                          # encoders + the counter commit
        self.vectors = self.streams * Lc * B * Hkv * 128
        self.Lc = Lc

    def reset(self):
        for w, t in zip((self.n_chunks, self.tail_start, self.tail_len), self.tmpl):
            w.copy_(t)

    def run(self):
        wl = self.wl
        self.tq.tq_evict(wl.kc, wl.vc, k_rec=self.krec, v_rec=self.vrec, k_tail=self.kt, v_tail=self.vt,
                         n_chunks=self.n_chunks, tail_start=self.tail_start, tail_len=self.tail_len,
                         window=EVICT_WINDOW, margin=EVICT_MARGIN, t_q=EVICT_TQ, max_evict=1)

    def run_layer(self, i: int):
        """The same call restricted to compressed layer i (the end-to-end leg's pipeline)."""
        wl, sl = self.wl, slice(i, i + 1)
        self.tq.tq_evict(wl.kc, wl.vc, k_rec=self.krec[sl], v_rec=self.vrec[sl], k_tail=self.kt[sl],
                         v_tail=self.vt[sl], n_chunks=self.n_chunks[sl], tail_start=self.tail_start[sl],
                         tail_len=self.tail_len[sl], window=EVICT_WINDOW, margin=EVICT_MARGIN, t_q=EVICT_TQ,
                         max_evict=1)

    def account(self):
        """Algorithmic bytes of one call: the evicted tokens read (bf16), the
        records written (codes, norms, counts and stored entries)."""
        torch, wl = self.torch, self.wl
        n = wl.n_rec - 1
        out = used_record_bytes(torch, self.krec[:, :, :, n], wl.kc, wl.d)
        if not wl.shared:
            out += used_record_bytes(torch, self.vrec[:, :, :, n], wl.vc, wl.d)
        self.bytes_in = self.vectors * wl.d * 2
        self.bytes_out = out
        self.bytes = self.bytes_in + self.bytes_out


class CacheWorkload:
    """A KV-cache workload.  One step = three phases, each replayed from its
    own CUDA graph and timed with CUDA events, L2 flushed before each:
      encode     tq_encode of every compressed layer's packed region (K and V)
      eviction   one tq_evict call moving one chunk per (layer, batch, kv head)
                 from the dense ring into its last record (EvictPhase)
      attention  one decode step of every layer in one tq_decode_attn call
                 over the records and the dense part (tail ring, or the
                 whole cache of a bf16 layer)."""

    def __init__(self, name, device, layers=None, batch=None, seed_offset: int = 0, splits: int = 0,
                 sparse_v: float = 0.0, sinks: bool = False):
        import torch

        import rotated_lloyd_max_gb300 as tq
        import synth
        self.tq, self.torch, self.dev, self.name = tq, torch, device, name
        cfg = dict(synth.CONFIGS[name])
        self.cfg = cfg
        L = layers or cfg["L"]
        B = batch or cfg["B"]
        Hkv, Hq, d, ctx = cfg["Hkv"], cfg["Hq"], cfg["d"], cfg["ctx"]
        self.L, self.B, self.Hkv, self.Hq, self.d, self.ctx = L, B, Hkv, Hq, d, ctx
        self.dense = [l for l in cfg.get("dense_layers", ()) if l < L]
        self.comp = [l for l in range(L) if l not in self.dense]
        assert self.comp == list(range(self.comp[0], self.comp[-1] + 1)), "compressed layers are contiguous"
        self.c0, self.c1 = self.comp[0], self.comp[-1] + 1
        tail = cfg.get("tail", 0)
        self.tail, self.n_rec = tail, (ctx - tail) // 128
        self.shared = cfg["shared_kv"]
        seed = cfg["data_seed"] + seed_offset
        T = cfg["T"]
        self.kc = tq.tq_make_codebook(cfg["kb"], d, sign_seed=cfg["sign_seed"], outlier_T=T)
        self.vc = self.kc if self.shared else tq.tq_make_codebook(cfg["vb"], d, sign_seed=cfg["sign_seed"],
                                                                  outlier_T=T)
        bf, u8, i32 = torch.bfloat16, torch.uint8, torch.int32
        # bf16 layers attend their whole cache as the dense part: their rows are ctx long
        ntok = ctx if self.dense else self.n_rec * 128
        self.ntok = ntok
        self.kx = torch.empty((L, B, Hkv, ntok, d), dtype=bf, device=device)
        self.vx = self.kx if self.shared else torch.empty_like(self.kx)
        self.q = torch.empty((L, B, Hq, d), dtype=bf, device=device)
        if tail:
            self.kt = torch.empty((L, B, Hkv, tail, d), dtype=bf, device=device)
            self.vt = self.kt if self.shared else torch.empty_like(self.kt)
        for l in range(L):
            synth.torch_gaussian_bf16(self.kx[l].shape, synth.layer_seed(seed, l, 0), device,
                                      out=self.kx[l], **synth.kv_recipe(cfg, "k"))
            if not self.shared:
                synth.torch_gaussian_bf16(self.vx[l].shape, synth.layer_seed(seed, l, 1), device,
                                          out=self.vx[l], **synth.kv_recipe(cfg, "v"))
            synth.torch_gaussian_bf16(self.q[l].shape, synth.layer_seed(seed, l, 2), device,
                                      scale=cfg["q_scale"], out=self.q[l])
            if tail:
                synth.torch_gaussian_bf16(self.kt[l].shape, synth.layer_seed(seed, l, 3), device,
                                          out=self.kt[l], **synth.kv_recipe(cfg, "k"))
                if not self.shared:
                    synth.torch_gaussian_bf16(self.vt[l].shape, synth.layer_seed(seed, l, 4), device,
                                              out=self.vt[l], **synth.kv_recipe(cfg, "v"))
        self.krec = torch.empty((L, B, Hkv, self.n_rec, self.kc.record_bytes), dtype=u8, device=device)
        self.vrec = self.krec if self.shared else torch.empty((L, B, Hkv, self.n_rec, self.vc.record_bytes),
                                                              dtype=u8, device=device)
        self.out = torch.empty((L, B, Hq, d), dtype=torch.float32, device=device)
        comp_mask = torch.tensor([l in self.comp for l in range(L)], device=device)[:, None].expand(L, B)
        self.n_chunks = torch.where(comp_mask, self.n_rec, 0).to(i32).contiguous()
        kw = dict(q=self.q, out=self.out, scale=1.0, k_rec=self.krec, v_rec=self.vrec, n_chunks=self.n_chunks,
                  max_chunks=self.n_rec, splits=splits)
        if self.dense:
            self.dense_len = torch.where(comp_mask, 0, ctx).to(i32).contiguous()
            kw.update(k_tail=self.kx, v_tail=self.vx, tail_len=self.dense_len, max_tail=ctx)
        elif tail:
            self.tail_len = torch.full((L, B), tail, dtype=i32, device=device)
            self.tail_start = torch.zeros((L, B), dtype=i32, device=device)
            kw.update(k_tail=self.kt, v_tail=self.vt, tail_len=self.tail_len, tail_start=self.tail_start,
                      max_tail=tail)
        self.args_all = tq.make_attn_args(**kw, sparse_v_eps=sparse_v)
        self.sparse_v = sparse_v
        if sparse_v:   # the same call without skipping, timed beside it
            self.args_exact = tq.make_attn_args(**kw)
        ws = tq.tq_decode_attn_workspace_size(self.args_all, self.kc, self.vc)
        self.args_layer = None
        if self.dense:          # the per-layer variant a model's layer loop issues (timed alongside)
            self.args_layer = []
            for l in range(L):
                if l in self.dense:
                    a = tq.make_attn_args(q=self.q[l:l + 1], out=self.out[l:l + 1], scale=1.0,
                                          k_tail=self.kx[l:l + 1], v_tail=self.vx[l:l + 1],
                                          tail_len=self.dense_len[l:l + 1], max_tail=ctx, splits=splits)
                    codecs = (None, None)
                else:
                    a = tq.make_attn_args(q=self.q[l:l + 1], out=self.out[l:l + 1], scale=1.0,
                                          k_rec=self.krec[l:l + 1], v_rec=self.vrec[l:l + 1],
                                          n_chunks=self.n_chunks[l:l + 1], max_chunks=self.n_rec, splits=splits)
                    codecs = (self.kc, self.vc)
                ws = max(ws, tq.tq_decode_attn_workspace_size(a, *codecs))
                self.args_layer.append((a, codecs))
        self.ws = torch.empty(ws, dtype=u8, device=device)
        self.plan = tq.tq_decode_attn_plan(self.args_all, self.kc, self.vc)
        self.sinks = sinks
        if sinks:
            self._plant_sinks()
        # eviction: the 144 tokens after the last record's are the dense tail's
        # first tokens where the workload has a tail, else a fresh draw
        lay = slice(self.c0, self.c1)
        Lc = self.c1 - self.c0
        if tail >= 144:
            nk = self.kt[lay, :, :, :144]
            nv = None if self.shared else self.vt[lay, :, :, :144]
        else:
            nk = torch.empty((Lc, B, Hkv, 144, d), dtype=bf, device=device)
            nv = None if self.shared else torch.empty_like(nk)
            for i in range(Lc):
                synth.torch_gaussian_bf16(nk[i].shape, synth.layer_seed(seed, self.c0 + i, 5), device, out=nk[i],
                                          **synth.kv_recipe(cfg, "k"))
                if nv is not None:
                    synth.torch_gaussian_bf16(nv[i].shape, synth.layer_seed(seed, self.c0 + i, 6), device,
                                              out=nv[i], **synth.kv_recipe(cfg, "v"))
        self.ev = EvictPhase(self, lay, nk, nv)
        del nk, nv
        # launches per step: one encode per stream, the eviction's, the attention call's
        streams = 1 if self.shared else 2
        self.enc_launches = streams
        self.launches_per_step = streams + self.ev.launches + self.plan["launches"]
        # algorithmic bytes (records counted as used: codes, norms, counts, stored entries)
        self.encode_k(); self.encode_v()
        self.ev.reset(); self.ev.run()
        torch.cuda.synchronize()
        self.ev.account()
        nc = len(self.comp)
        n_vec = nc * B * Hkv * self.n_rec * 128
        self.enc_in = streams * n_vec * d * 2
        self.enc_out = used_record_bytes(torch, self.krec[lay], self.kc, d) + (
            0 if self.shared else used_record_bytes(torch, self.vrec[lay], self.vc, d))
        dense_tok = len(self.dense) * B * Hkv * ctx + nc * B * Hkv * tail
        self.attn_bytes = (self.enc_out + streams * dense_tok * d * 2 + L * B * Hq * d * 2 + L * B * Hq * d * 4)
        # plain attention arithmetic: q.k and p.v per (query head, token), 2 flops per MAC
        self.attn_flops = 4 * L * B * Hq * d * ctx
        self.step_bytes = self.enc_in + self.enc_out + self.ev.bytes + self.attn_bytes
        self.concurrent_enc = self.enc_in < (256 << 20)
        self.vectors_per_step = streams * n_vec
        self.tokens_per_step = B          # one decode token per sequence through all layers

    def _plant_sinks(self):
        """A synthetic attention sink per block sequence of the decode kernel:
        the key u * 40 / min_h(q_h . u), u the sum of the kv head's queries, at
        token 128 r + 32 w of the first record r of every split, for each of
        the kernel's four warps w."""
        torch = self.torch
        cps = max(1, self.plan["records_per_split"])
        pos = torch.tensor([128 * r + 32 * w for r in range(0, self.n_rec, cps) for w in range(4)],
                           device=self.kx.device)
        G = self.Hq // self.Hkv
        for l in self.comp:
            q = self.q[l].float().view(self.B, self.Hkv, G, self.d)
            u = q.sum(2)                                                    # [B, Hkv, d]
            lo = torch.einsum("bhgd,bhd->bhg", q, u).amin(-1).clamp_min(1e-3)
            sink = (u * (40.0 / lo)[..., None]).to(torch.bfloat16)
            self.kx[l][:, :, pos] = sink[:, :, None, :]

    def attention_exact(self):
        self.tq.tq_decode_attn(self.args_exact, self.kc, self.vc, self.ws)

    def _enc(self, codec, src, rec):
        n = (self.c1 - self.c0) * self.B * self.Hkv
        nt = self.n_rec * 128
        self.tq.tq_encode(codec, src[self.c0:self.c1, :, :, :nt].view(n, nt, self.d),
                          rec[self.c0:self.c1].view(n, self.n_rec, -1))

    def encode_k(self):
        self._enc(self.kc, self.kx, self.krec)

    def encode_v(self):
        if not self.shared:
            self._enc(self.vc, self.vx, self.vrec)

    def encode_layer(self, l: int):
        """K and V encodes of one compressed layer (the end-to-end leg's pipeline)."""
        n = self.B * self.Hkv
        nt = self.n_rec * 128
        self.tq.tq_encode(self.kc, self.kx[l, :, :, :nt].reshape(n, nt, self.d), self.krec[l].view(n, self.n_rec, -1))
        if not self.shared:
            self.tq.tq_encode(self.vc, self.vx[l, :, :, :nt].reshape(n, nt, self.d),
                              self.vrec[l].view(n, self.n_rec, -1))

    def encode(self):
        """K and V encodes; when the cache is small (each launch a single wave
        that leaves most of the GPU idle) V's runs on a side stream, forked
        and joined through events."""
        if self.shared or not self.concurrent_enc:
            self.encode_k()
            self.encode_v()
            return
        torch = self.torch
        cur = torch.cuda.current_stream()
        if not hasattr(self, "_side"):
            self._side = torch.cuda.Stream()
            self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()
        self._fork.record(cur)
        self._side.wait_event(self._fork)
        self.encode_k()
        with torch.cuda.stream(self._side):
            self.encode_v()
        self._join.record(self._side)
        cur.wait_event(self._join)

    def attention(self):
        self.tq.tq_decode_attn(self.args_all, self.kc, self.vc, self.ws)

    def attention_per_layer(self):
        for a, (kc, vc) in self.args_layer:
            self.tq.tq_decode_attn(a, kc, vc, self.ws)

    def attention_layer(self, l: int):
        """Decode attention of compressed layer l alone (the end-to-end leg's
        pipeline: a layer's attention starts once its records are encoded)."""
        if not hasattr(self, "_args_comp"):
            self._args_comp = {}
            for c in self.comp:
                sl = slice(c, c + 1)
                kw = dict(q=self.q[sl], out=self.out[sl], scale=1.0, k_rec=self.krec[sl], v_rec=self.vrec[sl],
                          n_chunks=self.n_chunks[sl], max_chunks=self.n_rec)
                if self.tail:
                    kw.update(k_tail=self.kt[sl], v_tail=self.vt[sl], tail_len=self.tail_len[sl],
                              tail_start=self.tail_start[sl], max_tail=self.tail)
                a = self.tq.make_attn_args(**kw, sparse_v_eps=self.sparse_v)
                assert self.tq.tq_decode_attn_workspace_size(a, self.kc, self.vc) <= self.ws.numel()
                self._args_comp[c] = a
        self.tq.tq_decode_attn(self._args_comp[l], self.kc, self.vc, self.ws)

    def inputs(self):
        """Device tensors a step consumes from the host (leading axis: layer)."""
        d = {"kx": self.kx, "q": self.q, "evict_k": self.ev.kt}
        if not self.shared:
            d.update(vx=self.vx, evict_v=self.ev.vt)
        if self.tail:
            d["kt"] = self.kt
            if not self.shared:
                d["vt"] = self.vt
        return d

    def host_inputs(self):
        import numpy as np
        f = lambda t: t.contiguous().view(self.torch.int16).cpu().numpy().view(np.uint16)
        return {k: f(v) for k, v in (("kx", self.kx), ("vx", self.vx), ("q", self.q))}


def oracle_step(wl: CacheWorkload, hin: dict, layers=None):
    """The oracle on (a subset of) one step of a cache without a dense tail:
    encode the compressed layers' K/V, evict one chunk per stream (its
    encode), attend every listed layer.  Returns (algorithmic bytes, seconds)."""
    import oracle
    cfg = wl.cfg
    d, B, Hkv, Hq, ctx = wl.d, wl.B, wl.Hkv, wl.Hq, wl.ctx
    G = Hq // Hkv
    okc = oracle.Codec(d=d, bits=cfg["kb"], seed=cfg["sign_seed"])
    ovc = oracle.Codec(d=d, bits=cfg["vb"], seed=cfg["sign_seed"])
    layers = list(range(wl.L)) if layers is None else layers
    nbytes = 0
    t0 = time.perf_counter()
    for l in layers:
        for b in range(B):
            for h in range(Hkv):
                q = hin["q"][l, b, h * G:(h + 1) * G]
                if l in wl.dense:
                    oracle.unit_attention(q, None, None, None, None, 0, hin["kx"][l, b, h], hin["vx"][l, b, h], 1.0)
                    nbytes += 2 * ctx * d * 2
                else:
                    kr = oracle.encode_records(hin["kx"][l, b, h], okc)
                    vr = oracle.encode_records(hin["vx"][l, b, h], ovc)
                    ke = oracle.encode_records(hin["kx"][l, b, h, ctx - 128:], okc)
                    ve = oracle.encode_records(hin["vx"][l, b, h, ctx - 128:], ovc)
                    oracle.unit_attention(q, okc, ovc, kr, vr, ctx, None, None, 1.0)
                    nbytes += 2 * ctx * d * 2 + 2 * (kr.nbytes + vr.nbytes)
                    nbytes += 2 * 128 * d * 2 + ke.nbytes + ve.nbytes
                nbytes += G * d * 6
    return nbytes, time.perf_counter() - t0


# ---------------------------------------------------------------------------
# codec workloads: the round trip (tq_encode then tq_decode) and the encode sweep
# ---------------------------------------------------------------------------
def codec_items(cfg: dict) -> list:
    """(head dim, bit width) pairs a codec workload runs, in step order."""
    if cfg["kind"] == "codec":
        return [(cfg["d"], cfg["bits"])]
    return [(d, b) for d in cfg["ds"] for b in cfg["bits"]]


def codec_bytes(d: int, bits: int, n: int) -> dict:
    """Algorithmic bytes of encoding n bf16 vectors of head dim d at b bits
    (no outlier lists) and of decoding them to f32: encode reads 2d and writes
    d*b/8 code bytes + one f32 norm per vector; decode reads those record
    bytes and writes 4d per vector."""
    rec = n * (d * bits // 8 + 4)
    return {"enc_in": n * 2 * d, "enc_out": rec, "dec_in": rec, "dec_out": n * 4 * d}


class CodecWorkload:
    """The codec round trip (4096 x 128 vectors, N(0,1) x LogNormal(0, 0.5) per
    vector, b 3: tq_encode, then tq_decode of the records) and the encode sweep
    (2^24 N(0,1) vectors at each head dim 64..512 and bit width 2..4, one
    tq_encode each).  One step runs every item once; inputs, records and
    decoded rows stay in HBM."""

    def __init__(self, name, device):
        import torch

        import rotated_lloyd_max_gb300 as tq
        import synth
        self.tq, self.torch, self.name = tq, torch, name
        cfg = dict(synth.CONFIGS[name])
        self.cfg = cfg
        self.n = n = cfg["n"]
        self.with_decode = cfg["kind"] == "codec"
        self.src = {}
        for d in sorted({d for d, _ in codec_items(cfg)}):
            if self.with_decode:   # the round trip's parity inputs (host generator, seed 0)
                bits = synth.gaussian_bf16((n, d), cfg["data_seed"], lognormal_sigma=cfg["lognormal_sigma"])
                self.src[d] = torch.from_numpy(bits.view("int16")).view(torch.bfloat16).to(device)
            else:
                self.src[d] = synth.torch_gaussian_bf16((n, d), synth.layer_seed(cfg["data_seed"], d, 0), device)
        n_rec = (n + 127) // 128
        self.items = []
        for d, b in codec_items(cfg):
            c = tq.tq_make_codebook(b, d, sign_seed=cfg["sign_seed"])
            self.items.append({
                "d": d, "b": b, "codec": c,
                "rec": torch.empty((n_rec, c.record_bytes), dtype=torch.uint8, device=device),
                "dec": torch.empty((n, d), dtype=torch.float32, device=device) if self.with_decode else None,
                **codec_bytes(d, b, n)})
        self.launches_per_step = len(self.items) * (2 if self.with_decode else 1)
        self.enc_bytes = sum(it["enc_in"] + it["enc_out"] for it in self.items)
        self.dec_bytes = sum(it["dec_in"] + it["dec_out"] for it in self.items) if self.with_decode else 0
        self.step_bytes = self.enc_bytes + self.dec_bytes

    def encode(self, it):
        self.tq.tq_encode(it["codec"], self.src[it["d"]], it["rec"])

    def decode(self, it):
        self.tq.tq_decode(it["codec"], it["rec"], it["dec"])

    def step(self):
        for it in self.items:
            self.encode(it)
            if self.with_decode:
                self.decode(it)


def run_codec(args, world, rank, local, pg):
    """Timed steps of a codec workload: each kernel launch bracketed by CUDA
    events on the launching stream, L2 flushed before every step (the sweep's
    inputs, 2-16 GiB per item, exceed L2 on their own)."""
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rotated_lloyd_max_gb300 import build as b
    b.build()
    import rotated_lloyd_max_gb300 as tq
    tq.load()
    wl = CodecWorkload(args.workload, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize()
    # every launch is captured once and replayed: the round trip's kernels run
    # for microseconds, less than the host's argument marshalling per call
    graphs = []
    for it in wl.items:
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, capture_error_mode="relaxed"):
            wl.encode(it)
        gd = None
        if wl.with_decode:
            gd = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gd, capture_error_mode="relaxed"):
                wl.decode(it)
        graphs.append((ge, gd))
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        for ge, gd in graphs:
            ge.replay()
            if gd is not None:
                gd.replay()
    torch.cuda.synchronize()
    K = args.steps
    n_it = len(wl.items)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_it)] for _ in range(K)]
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    barrier(pg)
    torch.cuda.synchronize()
    for s in range(K):
        flush.zero_()
        for i, (ge, gd) in enumerate(graphs):
            e = ev[s][i]
            e[0].record(stream)
            ge.replay()
            e[1].record(stream)
            if gd is not None:
                gd.replay()
            e[2].record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    t_enc = [[ev[s][i][0].elapsed_time(ev[s][i][1]) / 1e3 for s in range(K)] for i in range(n_it)]
    t_dec = [[ev[s][i][1].elapsed_time(ev[s][i][2]) / 1e3 for s in range(K)] for i in range(n_it)]
    total = sum(map(sum, t_enc)) + (sum(map(sum, t_dec)) if wl.with_decode else 0.0)
    total_max = max_over_ranks(pg, total, dev)
    bytes_all = sum_over_ranks(pg, wl.step_bytes * K, dev)
    value = bytes_all / total_max / 1e9
    hbm, _, peak_kind = peaks()
    enc_s, dec_s = sum(map(sum, t_enc)) / K, sum(map(sum, t_dec)) / K
    dominant = "tq_decode" if wl.with_decode and dec_s > enc_s else "tq_encode"
    dom_bytes, dom_s = (wl.dec_bytes, dec_s) if dominant == "tq_decode" else (wl.enc_bytes, enc_s)
    achieved = dom_bytes / dom_s / 1e9            # = bytes per launch / mean launch time, summed over items
    per_item = []
    for i, it in enumerate(wl.items):
        te = sum(t_enc[i]) / K
        row = {"d": it["d"], "bits": it["b"], "encode_us": round(te * 1e6, 2),
               "encode_gbs": round((it["enc_in"] + it["enc_out"]) / te / 1e9, 1),
               "encode_frac": round((it["enc_in"] + it["enc_out"]) / te / 1e9 / hbm, 4)}
        if wl.with_decode:
            td = sum(t_dec[i]) / K
            row.update({"decode_us": round(td * 1e6, 2),
                        "decode_gbs": round((it["dec_in"] + it["dec_out"]) / td / 1e9, 1)})
        per_item.append(row)
    line = {
        "metric": "decode-attn KV GB/s & tok/s; encode Mvec/s; % of GB300 HBM roofline",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_max / K * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, packed codes, f32 math" + (", f32 out" if wl.with_decode else ""),
        "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "vectors": wl.n,
                   "items": [f"d{d}/b{b}" for d, b in codec_items(wl.cfg)],
                   "step": "tq_encode" + (" then tq_decode" if wl.with_decode else "") + " of every item",
                   "l2": "flushed (256 MiB write) before each step", "parallelism": f"replicas x{world}"},
        "breakdown": {"encode_mvec_s": round(wl.n * n_it / enc_s / 1e6, 1),
                      "encode_gbs": round(wl.enc_bytes / enc_s / 1e9, 1),
                      **({"decode_gbs": round(wl.dec_bytes / dec_s / 1e9, 1)} if wl.with_decode else {}),
                      "items": per_item, "step_algorithmic_bytes": wl.step_bytes},
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "per_step_bytes": dom_bytes,
                     "traffic": None},
        "gpu_launches": wl.launches_per_step * K,
    }
    if clk:
        line["clocks"] = clk
    if not args.no_e2e:
        line["e2e"] = codec_e2e(wl, max(3, min(20, K)))
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        nbytes, secs, sample = codec_oracle_sample(wl.cfg)
        import oracle
        line["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s",
                                "cores": oracle.threads(), "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)


def codec_e2e(wl, steps: int):
    """The codec step through the public API with host buffers: each item's
    bf16 rows copied in from pinned memory, encoded (and decoded), and its
    product (decoded rows, or the records) copied back, all timed."""
    import torch
    pin_in = {d: t.cpu().pin_memory() for d, t in wl.src.items()}
    prod = [it["dec"] if wl.with_decode else it["rec"] for it in wl.items]
    pin_out = [torch.empty(p.shape, dtype=p.dtype).pin_memory() for p in prod]
    h2d = sum(t.numel() * t.element_size() for t in pin_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pin_out)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        for d, t in pin_in.items():
            wl.src[d].copy_(t, non_blocking=True)
        for it, p, h in zip(wl.items, prod, pin_out):
            wl.encode(it)
            if wl.with_decode:
                wl.decode(it)
            h.copy_(p, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    secs = (time.perf_counter() - t0) / steps
    return {"value": round(wl.step_bytes / secs / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3, 4)}


def codec_oracle_sample(cfg: dict, n_max: int = 4096):
    """The oracle (fp64 C) on the workload's items with at most n_max vectors
    each (the round trip in full): (algorithmic bytes, seconds, description)."""
    import oracle
    import synth
    oracle.build()
    n = min(cfg["n"], n_max)
    decode = cfg["kind"] == "codec"
    nbytes, secs = 0, 0.0
    for d, b in codec_items(cfg):
        if decode:
            x = synth.gaussian_bf16((n, d), cfg["data_seed"], lognormal_sigma=cfg["lognormal_sigma"])
        else:
            x = synth.gaussian_bf16((n, d), synth.layer_seed(cfg["data_seed"], d, 0))
        oc = oracle.Codec(d=d, bits=b, seed=cfg["sign_seed"])
        t0 = time.perf_counter()
        rec = oracle.encode_records(x, oc)
        if decode:
            oracle.decode_records(rec, n, oc)
        secs += time.perf_counter() - t0
        by = codec_bytes(d, b, n)
        nbytes += by["enc_in"] + by["enc_out"] + ((by["dec_in"] + by["dec_out"]) if decode else 0)
    what = "encode + decode" if decode else "encode"
    return nbytes, secs, f"{what} of {n} vectors per item ({len(codec_items(cfg))} items), fp64 C oracle"


WORKLOADS = {"qwen2_1p5b_ctx2048": CacheWorkload,
             "batched_b32_ctx32768": CacheWorkload,
             "v4flash_mqa_ctx65536": CacheWorkload,
             "longctx_b4_ctx262144": CacheWorkload,
             "codec_roundtrip_4096x128_b3": CodecWorkload,
             "encode_sweep_16M": CodecWorkload}


def roofline_entry(kernel: str, nbytes: int, secs: float, launches: int, flops: int | None = None):
    """The roofline of one phase: algorithmic bytes (or flops) per step over
    the phase's CUDA-event time; attention whose plain arithmetic intensity
    exceeds the ridge point is reported against the tensor peak."""
    hbm, tflops, peak_kind = peaks()
    gbs = nbytes / secs / 1e9
    e = {"kernel": kernel, "launches_per_step": launches}
    ridge = tflops * 1e12 / (hbm * 1e9)
    if flops is not None and flops / nbytes > ridge:
        tf = flops / secs / 1e12
        e.update({"bound": "tensor", "achieved": round(tf, 2), "peak": tflops, "unit": "TFLOP/s",
                  "frac": round(tf / tflops, 4),
                  "peak_kind": f"{peak_kind} dense bf16 GEMM (burst); the kernel's f16 MMAs run at the same rate",
                  "per_step_flops": flops, "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)})
    else:
        e.update({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(gbs / hbm, 4), "peak_kind": f"{peak_kind} HBM copy bandwidth"})
    e["per_step_bytes"] = nbytes
    if flops is not None:
        e.update({"intensity_flop_per_byte": round(flops / nbytes, 1), "ridge_flop_per_byte": round(ridge, 1)})
    e["time_us"] = round(secs * 1e6, 2)
    return e


def run_native(args, world, rank, local, pg):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rotated_lloyd_max_gb300 import build as b
    b.build()
    import rotated_lloyd_max_gb300 as tq
    tq.load()
    wl = CacheWorkload(args.workload, dev, layers=args.layers, batch=args.batch, splits=args.splits,
                       sparse_v=args.sparse_v, sinks=args.sinks)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step_eager():
        flush.zero_(); wl.encode()
        wl.ev.reset(); flush.zero_(); wl.ev.run()
        flush.zero_(); wl.attention()

    for _ in range(max(args.warmup, 3)):
        step_eager()
    torch.cuda.synchronize()
    # each phase is captured once and replayed, so the timed region measures
    # device work, not the host's per-call argument marshalling
    graphs = []
    for fn in (wl.encode, wl.ev.reset, wl.ev.run, wl.attention):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn()
        graphs.append(g)
    g_enc, g_reset, g_ev, g_attn = graphs

    def step(e=None):
        flush.zero_()
        if e: e[0].record(stream)
        g_enc.replay()
        if e: e[1].record(stream)
        g_reset.replay()                  # counter templates (three 4-byte-per-unit copies), untimed
        flush.zero_()
        if e: e[2].record(stream)
        g_ev.replay()
        if e: e[3].record(stream)
        flush.zero_()
        if e: e[4].record(stream)
        g_attn.replay()
        if e: e[5].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    barrier(pg)
    torch.cuda.synchronize()
    for s in range(K):
        step(ev[s])
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    t_enc = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3 / K
    t_ev = sum(e[2].elapsed_time(e[3]) for e in ev) / 1e3 / K
    t_attn = sum(e[4].elapsed_time(e[5]) for e in ev) / 1e3 / K
    total = (t_enc + t_ev + t_attn) * K
    total_max = max_over_ranks(pg, total, dev)
    bytes_all = sum_over_ranks(pg, wl.step_bytes * K, dev)
    value = bytes_all / total_max / 1e9
    phases = {
        "tq_encode": roofline_entry("tq_encode" + ("" if wl.shared else " (K and V concurrent on two streams)"
                                                   if wl.concurrent_enc else " (K then V)"),
                                    wl.enc_in + wl.enc_out, t_enc, wl.enc_launches),
        "tq_evict": roofline_entry("tq_evict (one chunk per layer, batch and kv head)", wl.ev.bytes, t_ev,
                                   wl.ev.launches),
        "tq_decode_attn": roofline_entry(f"tq_decode_attn ({wl.plan['compressed_kernel']} + "
                                         f"{wl.plan['dense_kernel']} dense splits + merge)",
                                         wl.attn_bytes, t_attn, wl.plan["launches"], flops=wl.attn_flops),
    }
    for name, e in phases.items():
        full = wl.L == wl.cfg["L"] and wl.B == wl.cfg["B"] and not wl.sparse_v and not wl.sinks
        t = measured_traffic(wl.name if full else "", name)
        e["traffic"] = t
        e["traffic_sources_sha"] = phase_sources_sha(name)
    dominant = max(phases, key=lambda k: phases[k]["time_us"])
    per_layer = per_layer_attention(wl, stream, flush, max(3, min(200, K))) if wl.args_layer else None
    exact_attn = exact_attention_time(wl, stream, flush, K) if wl.sparse_v else None
    cfg = wl.cfg
    line = {
        "metric": "decode-attn KV GB/s & tok/s; encode Mvec/s; % of GB300 HBM roofline",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_max / K * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, packed codes, f32 math",
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": wl.name, "layers": wl.L, "batch": wl.B, "kv_heads": wl.Hkv,
                   "q_heads": wl.Hq, "head_dim": wl.d, "ctx": wl.ctx, "k_bits": cfg["kb"],
                   "v_bits": cfg["vb"], "outlier_T": cfg["T"], "bf16_layers": wl.dense,
                   "tail_tokens": wl.tail, "full_size": wl.L == cfg["L"] and wl.B == cfg["B"],
                   "l2": "flushed (256 MiB write) before each phase, outside its events",
                   "attention_splits": args.splits or "planner",
                   **({"sparse_v_eps": wl.sparse_v} if wl.sparse_v else {}),
                   **({"sinks": "attention-sink key at the first token of each warp block opening a split"}
                      if wl.sinks else {}),
                   "step": (f"encode whole cache ({wl.enc_launches} launch(es)) + evict one chunk per "
                            f"(layer, batch, kv head) ({wl.ev.launches} launches) + decode attention of all "
                            f"{wl.L} layers in one tq_decode_attn call ({wl.plan['launches']} launches)"),
                   "eviction": {"window": EVICT_WINDOW, "margin": EVICT_MARGIN, "t_q": EVICT_TQ,
                                "ring_slots": wl.ev.cap, "chunks_per_call": 1},
                   "parallelism": f"replicas x{world}"},
        "breakdown": {
            "encode_mvec_s": round(wl.vectors_per_step / t_enc / 1e6, 1),
            "encode_us_per_step": round(t_enc * 1e6, 2),
            "evict_mvec_s": round(wl.ev.vectors / t_ev / 1e6, 1),
            "evict_us_per_step": round(t_ev * 1e6, 2),
            "decode_attn_kv_gbs": round(wl.attn_bytes / t_attn / 1e9, 1),
            "decode_attn_tok_s": round(wl.tokens_per_step / t_attn, 1),
            "decode_attn_us_per_step": round(t_attn * 1e6, 2),
            **({"decode_attn_per_layer_calls_us_per_step": round(per_layer * 1e6, 2)} if per_layer else {}),
            **({"sparse_v": {"eps": wl.sparse_v, "decode_attn_us_per_step": round(t_attn * 1e6, 2),
                             "decode_attn_us_per_step_without": round(exact_attn * 1e6, 2)}}
               if wl.sparse_v else {}),
            "step_algorithmic_bytes": wl.step_bytes,
            "attention_plan": wl.plan,
        },
        "roofline": {**phases[dominant], "phase": dominant},
        "roofline_phases": phases,
        "gpu_launches": wl.launches_per_step * K,
    }
    if clk:
        line["clocks"] = clk
    if not args.no_e2e:
        line["e2e"] = e2e_leg(wl, max(3, min(50 if wl.step_bytes < (1 << 30) else 3, K)))
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        import oracle
        if wl.dense:
            hin = wl.host_inputs()
            nbytes, secs = oracle_step(wl, hin)
            sample = (f"one full step (all {wl.L} layers: encode of the {len(wl.comp)} compressed layers, one "
                      "evicted chunk per stream, attention of every layer), fp64 C oracle")
        else:
            step_o, sample = oracle_unit_sample(wl.cfg)
            step_o()                                   # warm-up
            t0 = time.perf_counter()
            nbytes = step_o()
            secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s",
                                "cores": oracle.threads(), "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)


def exact_attention_time(wl, stream, flush, steps: int) -> float:
    """The attention call without sparse-V skipping, replayed from a CUDA graph
    with L2 flushed before each replay; mean seconds."""
    import torch
    graph = torch.cuda.CUDAGraph()
    wl.attention_exact()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        wl.attention_exact()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b) / 1e3
    return tot / steps


def per_layer_attention(wl, stream, flush, steps: int) -> float:
    """Decode attention as per-layer tq_decode_attn calls replayed from a CUDA
    graph (the shape a model's layer loop issues); mean seconds per step."""
    import torch
    graph = torch.cuda.CUDAGraph()
    wl.attention_per_layer()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        wl.attention_per_layer()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b) / 1e3
    return tot / steps


E2E_PIN_LIMIT = 2 << 30   # larger inputs are staged from one pinned layer slice
E2E_PIPELINE_MIN = 1 << 30  # from this many bytes of inputs per step, copies overlap the layer encodes


def e2e_leg(wl, steps: int):
    """The step through the public API with host buffers: every input of the
    step (the bf16 K/V the encode reads, the ring tokens the eviction reads,
    q and the dense tail) copied in from pinned host memory, the three phases
    run, the attention output copied back, all inside the timed region.  An
    input larger than 2 GiB is copied layer by layer from one pinned
    layer-sized host buffer (every layer receives the same host bytes: the
    copied volume is the full input, the host memory pinned is one layer).
    From 1 GiB of inputs per step the copies run on a copy stream, layer by
    layer, and each compressed layer is encoded, evicted and attended as soon
    as its inputs have arrived (one tq_evict and one tq_decode_attn call per
    layer, as a model's layer loop issues them), so all three phases overlap
    the later layers' copies; bf16 layers are attended once every copy is in.
    Smaller steps copy everything first and then run the step (per-layer
    launches would dominate them)."""
    import torch
    srcs = wl.inputs()
    pipelined = sum(t.numel() * t.element_size() for t in srcs.values()) >= E2E_PIPELINE_MIN
    # inputs copied layer by layer, and the absolute layer of their index 0 (the
    # pipeline also takes each layer's ring and tail tokens with its K/V)
    layer_axis = {"kx": 0, "vx": 0}
    if pipelined:
        layer_axis.update(kt=0, vt=0, evict_k=wl.c0, evict_v=wl.c0)
    small, per_layer = [], [[] for _ in range(wl.L)]
    for name, t in srcs.items():
        big = t.numel() * t.element_size() > E2E_PIN_LIMIT
        if name in layer_axis:
            h = t[0].cpu().pin_memory() if big else t.cpu().pin_memory()
            for i in range(t.shape[0]):
                per_layer[layer_axis[name] + i].append((t[i], h if big else h[i]))
        elif big:
            h = t[0].cpu().pin_memory()
            small += [(t[l], h) for l in range(t.shape[0])]
        else:
            small.append((t, t.cpu().pin_memory()))
    out_h = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()
    h2d = sum(dv.numel() * dv.element_size() for dv, _ in small + [x for lay in per_layer for x in lay])
    d2h = out_h.numel() * out_h.element_size()
    cur = torch.cuda.current_stream()
    if not pipelined:
        # a small step: copies and the whole-cache encode back to back (a
        # per-layer pipeline would be launch-bound)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            for dv, h in [x for lay in per_layer for x in lay] + small:
                dv.copy_(h, non_blocking=True)
            wl.encode()
            wl.ev.reset(); wl.ev.run()
            wl.attention()
            out_h.copy_(wl.out, non_blocking=True)
            cur.synchronize()
        secs = (time.perf_counter() - t0) / steps
        return {"value": round(wl.step_bytes / secs / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3, 4),
                "pipeline": "copies, then the step (inputs below 1 GiB)"}
    copy = torch.cuda.Stream()
    arrived = [torch.cuda.Event() for _ in range(wl.L)]
    start, first = torch.cuda.Event(), torch.cuda.Event()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        start.record(cur)
        copy.wait_event(start)
        with torch.cuda.stream(copy):
            for dv, h in small:                      # q and other small inputs first
                dv.copy_(h, non_blocking=True)
            first.record(copy)
            for l in range(wl.L):
                for dv, h in per_layer[l]:
                    dv.copy_(h, non_blocking=True)
                arrived[l].record(copy)
        cur.wait_event(first)
        wl.ev.reset()
        for l in wl.comp:
            cur.wait_event(arrived[l])
            wl.encode_layer(l)
            wl.ev.run_layer(l - wl.c0)
            wl.attention_layer(l)
        if wl.dense:
            cur.wait_event(arrived[wl.L - 1])
            for a, (kc, vc) in [wl.args_layer[l] for l in wl.dense]:
                wl.tq.tq_decode_attn(a, kc, vc, wl.ws)
        out_h.copy_(wl.out, non_blocking=True)
        cur.synchronize()
    secs = (time.perf_counter() - t0) / steps
    return {"value": round(wl.step_bytes / secs / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3, 4),
            "pipeline": "layer copies on a copy stream; each layer encoded, evicted and attended on arrival"}


def oracle_unit_sample(cfg: dict):
    """The oracle's bounded sample of a cache workload: one (layer, kv head)
    unit of a compressed layer (its packed tokens encoded, one record stream
    when keys and values share records; its last chunk encoded again as the
    eviction phase does; then attended with the unit's dense tail) plus one
    unit of a bf16 layer where the workload has them.
    Returns (step() -> algorithmic bytes, description)."""
    import oracle
    import synth
    oracle.build()
    d, ctx, Hkv, Hq = cfg["d"], cfg["ctx"], cfg["Hkv"], cfg["Hq"]
    G = Hq // Hkv
    T, shared, tail = cfg["T"], cfg["shared_kv"], cfg.get("tail", 0)
    nc = (ctx - tail) // 128 * 128                                   # tokens held in records
    okc = oracle.Codec(d=d, bits=cfg["kb"], seed=cfg["sign_seed"], T=T)
    ovc = okc if shared else oracle.Codec(d=d, bits=cfg["vb"], seed=cfg["sign_seed"], T=T)
    seed = cfg["data_seed"]
    k = synth.gaussian_bf16((ctx, d), synth.layer_seed(seed, 3, 0), **synth.kv_recipe(cfg, "k"))
    v = k if shared else synth.gaussian_bf16((ctx, d), synth.layer_seed(seed, 3, 1))
    q = synth.gaussian_bf16((G, d), synth.layer_seed(seed, 3, 2), scale=cfg["q_scale"])
    dense = bool(cfg["dense_layers"])
    if dense:
        kd = synth.gaussian_bf16((ctx, d), synth.layer_seed(seed, 0, 0), **synth.kv_recipe(cfg, "k"))
        vd = synth.gaussian_bf16((ctx, d), synth.layer_seed(seed, 0, 1))
    streams = 1 if shared else 2

    def step():
        kr = oracle.encode_records(k[:nc], okc)
        vr = kr if shared else oracle.encode_records(v[:nc], ovc)
        ke = oracle.encode_records(k[nc - 128:nc], okc)
        ve = ke if shared else oracle.encode_records(v[nc - 128:nc], ovc)
        kt, vt = (k[nc:], v[nc:]) if tail else (None, None)
        oracle.unit_attention(q, okc, ovc, kr, vr, nc, kt, vt, 1.0)
        rec = kr.nbytes + (0 if shared else vr.nbytes)
        nb = streams * nc * d * 2 + rec                              # encode: bf16 in, records out
        nb += streams * 128 * d * 2 + ke.nbytes + (0 if shared else ve.nbytes)   # eviction of one chunk
        nb += rec + streams * tail * d * 2 + G * d * 6               # attention: records, tail, q, out
        if dense:
            oracle.unit_attention(q, None, None, None, None, 0, kd, vd, 1.0)
            nb += 2 * ctx * d * 2 + G * d * 6
        return nb
    sample = (f"one (layer, kv head) unit ({nc} packed tokens, {streams} stream(s), its last chunk evicted "
              f"again) attended with its {tail}-token dense tail" + (", plus one bf16-layer unit" if dense else "")
              + ", fp64 C oracle")
    return step, sample


def run_reference(args, world, rank, local, pg):
    """The oracle (fp64 C, OpenMP) on the host cores: each step encodes one
    (layer, kv head) unit of a compressed layer (its packed tokens, one record
    stream when keys and values share records) and attends it with the unit's
    dense tail, plus one unit of a bf16 layer where the workload has them, so
    K steps finish within minutes."""
    if rank != 0:
        return
    import oracle
    import synth
    cfg = synth.CONFIGS[args.workload]
    step, sample = oracle_unit_sample(cfg)

    budget = 150.0
    for _ in range(max(args.warmup, 3) if args.warmup < 1000 else 3):
        step()
    t0 = time.perf_counter()
    nbytes = step()
    one = time.perf_counter() - t0
    K = args.steps
    n_run = K if one * K <= budget else max(1, int(budget / one))
    t0 = time.perf_counter()
    total = 0
    for _ in range(n_run):
        total += step()
    secs = time.perf_counter() - t0
    value = total / secs / 1e9
    line = {
        "impl": "reference",
        "metric": "decode-attn KV GB/s & tok/s; encode Mvec/s; % of GB300 HBM roofline",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(secs / n_run * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "sample": "per step: " + sample, "steps_run": n_run},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{n_run} steps of: " + sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_codec(args, world, rank, local, pg):
    """The oracle on a codec workload: each step encodes (and for the round
    trip decodes) at most 4096 vectors of every item, on the host cores."""
    if rank != 0:
        return
    import oracle
    import synth
    cfg = synth.CONFIGS[args.workload]
    for _ in range(min(max(args.warmup, 3), 3)):
        codec_oracle_sample(cfg)
    budget = 150.0
    nbytes, one, sample = codec_oracle_sample(cfg)
    K = args.steps
    n_run = K if one * K <= budget else max(1, int(budget / one))
    total, secs = 0, 0.0
    for _ in range(n_run):
        b, t, _ = codec_oracle_sample(cfg)
        total += b
        secs += t
    value = total / secs / 1e9
    line = {
        "impl": "reference",
        "metric": "decode-attn KV GB/s & tok/s; encode Mvec/s; % of GB300 HBM roofline",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(secs / n_run * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "sample": sample, "steps_run": n_run},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{n_run} steps: {sample}"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.steps is None:
        args.steps = {"qwen2_1p5b_ctx2048": 5000, "codec_roundtrip_4096x128_b3": 2000,
                      "encode_sweep_16M": 5}.get(args.workload, 20)
    world, rank, local, pg = dist_init(args.gpus)
    try:
        codec = WORKLOADS[args.workload] is CodecWorkload
        if args.impl == "reference":
            (run_reference_codec if codec else run_reference)(args, world, rank, local, pg)
        else:
            (run_codec if codec else run_native)(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    main()
