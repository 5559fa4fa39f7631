#!/usr/bin/env python
"""Benchmark of the rotated Lloyd-Max KV-cache path on GB300.

Default workload: the Qwen2-1.5B-shaped cache (28 layers, 2 KV heads, 12 query
heads, head_dim 128, batch 1, ctx 2048; K 3 bits, V 2 bits; layers 0-2 and
25-27 kept bf16).  One step = encode the whole compressed cache (K and V of 22
layers, two tq_encode launches) + one decode step of tq_decode_attn per layer
(28 calls, replayed from a CUDA graph).  Inputs are synthetic, generated on the
device from fixed seeds, resident in HBM before timing.  L2 is flushed (a
256 MiB write) before every timed step; each step is timed with CUDA events.

value = algorithmic HBM bytes of the step (bytes each kernel must read and
write by the record layout) / device time, in GB/s.  Also reported: encode
Mvec/s, decode-attention KV GB/s and tok/s, the roofline of the dominant kernel
against the measured HBM copy bandwidth, the oracle (CPU) timed on a bounded
sample, and an end-to-end figure with host buffers copied in and out.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload qwen2_1p5b_ctx2048|batched_b32_ctx32768|v4flash_mqa_ctx65536|longctx_b4_ctx262144]
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
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="qwen2_1p5b_ctx2048")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class QwenCache:
    """Qwen2-1.5B-shaped cache: encode the whole cache, then one decode step of
    tq_decode_attn per layer."""

    name = "qwen2_1p5b_ctx2048"

    def __init__(self, device, seed_offset: int = 0):
        import torch

        import rotated_lloyd_max_gb300 as tq
        import synth
        self.tq, self.torch, self.dev = tq, torch, device
        cfg = dict(synth.CONFIGS[self.name])
        self.cfg = cfg
        L, B, Hkv, Hq, d, ctx = cfg["L"], cfg["B"], cfg["Hkv"], cfg["Hq"], cfg["d"], cfg["ctx"]
        self.L, self.B, self.Hkv, self.Hq, self.d, self.ctx = L, B, Hkv, Hq, d, ctx
        self.dense = list(cfg["dense_layers"])
        self.comp = [l for l in range(L) if l not in self.dense]
        nc, nd = len(self.comp), len(self.dense)
        seed = cfg["data_seed"] + seed_offset
        self.kc = tq.tq_make_codebook(cfg["kb"], d, sign_seed=cfg["sign_seed"])
        self.vc = tq.tq_make_codebook(cfg["vb"], d, sign_seed=cfg["sign_seed"])
        bf = torch.bfloat16
        self.k_src = torch.empty((nc, B, Hkv, ctx, d), dtype=bf, device=device)
        self.v_src = torch.empty_like(self.k_src)
        self.k_dense = torch.empty((nd, B, Hkv, ctx, d), dtype=bf, device=device)
        self.v_dense = torch.empty_like(self.k_dense)
        for i, l in enumerate(self.comp):
            synth.torch_gaussian_bf16(self.k_src[i].shape, synth.layer_seed(seed, l, 0), device,
                                      fixed_channels=cfg["k_fixed_channels"], out=self.k_src[i])
            synth.torch_gaussian_bf16(self.v_src[i].shape, synth.layer_seed(seed, l, 1), device,
                                      out=self.v_src[i])
        for i, l in enumerate(self.dense):
            synth.torch_gaussian_bf16(self.k_dense[i].shape, synth.layer_seed(seed, l, 0), device,
                                      fixed_channels=cfg["k_fixed_channels"], out=self.k_dense[i])
            synth.torch_gaussian_bf16(self.v_dense[i].shape, synth.layer_seed(seed, l, 1), device,
                                      out=self.v_dense[i])
        self.q = torch.empty((L, B, Hq, d), dtype=bf, device=device)
        for l in range(L):
            synth.torch_gaussian_bf16(self.q[l].shape, synth.layer_seed(seed, l, 2), device,
                                      scale=cfg["q_scale"], out=self.q[l])
        self.n_rec = ctx // 128
        self.krec = torch.empty((nc, B, Hkv, self.n_rec, self.kc.record_bytes), dtype=torch.uint8, device=device)
        self.vrec = torch.empty((nc, B, Hkv, self.n_rec, self.vc.record_bytes), dtype=torch.uint8, device=device)
        self.out = torch.empty((L, B, Hq, d), dtype=torch.float32, device=device)
        i32 = torch.int32
        self.n_chunks = torch.full((nc, B), self.n_rec, dtype=i32, device=device)
        self.ctx_len = torch.full((nd, B), ctx, dtype=i32, device=device)
        # per-layer argument blocks, built once (pointers are fixed)
        self.args = []
        ws = 0
        for l in range(L):
            if l in self.dense:
                j = self.dense.index(l)
                a = tq.make_attn_args(q=self.q[l:l + 1], out=self.out[l:l + 1], scale=1.0,
                                      k_tail=self.k_dense[j:j + 1], v_tail=self.v_dense[j:j + 1],
                                      tail_len=self.ctx_len[j:j + 1], max_tail=ctx)
                codecs = (None, None)
            else:
                i = self.comp.index(l)
                a = tq.make_attn_args(q=self.q[l:l + 1], out=self.out[l:l + 1], scale=1.0,
                                      k_rec=self.krec[i:i + 1], v_rec=self.vrec[i:i + 1],
                                      n_chunks=self.n_chunks[i:i + 1], max_chunks=self.n_rec)
                codecs = (self.kc, self.vc)
            ws = max(ws, tq.tq_decode_attn_workspace_size(a, *codecs))
            self.args.append((a, codecs))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.launches_per_step = 2 + 2 * L
        # algorithmic bytes
        d2 = d * 2
        n_vec_stream = nc * B * Hkv * ctx
        self.enc_in = 2 * n_vec_stream * d2
        self.enc_out = nc * B * Hkv * self.n_rec * (self.kc.record_bytes + self.vc.record_bytes)
        self.attn_bytes = (self.enc_out + nd * B * Hkv * ctx * 2 * d2 + L * B * Hq * d * 2
                           + L * B * Hq * d * 4)
        self.step_bytes = self.enc_in + self.enc_out + self.attn_bytes
        self.vectors_per_step = 2 * n_vec_stream
        self.tokens_per_step = B  # one decode token per sequence through all layers

    # encode launches (timed with events individually)
    def encode_k(self):
        nc, B, Hkv = len(self.comp), self.B, self.Hkv
        self.tq.tq_encode(self.kc, self.k_src.view(nc * B * Hkv, self.ctx, self.d),
                          self.krec.view(nc * B * Hkv, self.n_rec, -1))

    def encode_v(self):
        nc, B, Hkv = len(self.comp), self.B, self.Hkv
        self.tq.tq_encode(self.vc, self.v_src.view(nc * B * Hkv, self.ctx, self.d),
                          self.vrec.view(nc * B * Hkv, self.n_rec, -1))

    def attention(self):
        for a, (kc, vc) in self.args:
            self.tq.tq_decode_attn(a, kc, vc, self.ws)

    # host copies for the oracle / end-to-end leg
    def host_inputs(self):
        import numpy as np
        f = lambda t: t.contiguous().view(self.torch.int16).cpu().numpy().view(np.uint16)
        return dict(k_src=f(self.k_src), v_src=f(self.v_src), k_dense=f(self.k_dense), v_dense=f(self.v_dense),
                    q=f(self.q))


def oracle_step(wl: QwenCache, hin: dict, layers=None):
    """The oracle on (a subset of) one step: encode the compressed layers' K/V
    and attend every listed layer.  Returns (algorithmic bytes, seconds)."""
    import numpy as np

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
                    j = wl.dense.index(l)
                    oracle.unit_attention(q, None, None, None, None, 0, hin["k_dense"][j, b, h],
                                          hin["v_dense"][j, b, h], 1.0)
                    nbytes += 2 * ctx * d * 2
                else:
                    i = wl.comp.index(l)
                    kr = oracle.encode_records(hin["k_src"][i, b, h], okc)
                    vr = oracle.encode_records(hin["v_src"][i, b, h], ovc)
                    oracle.unit_attention(q, okc, ovc, kr, vr, ctx, None, None, 1.0)
                    nbytes += 2 * ctx * d * 2 + 2 * (kr.nbytes + vr.nbytes)
                nbytes += G * d * 6
    return nbytes, time.perf_counter() - t0


WORKLOADS = {"qwen2_1p5b_ctx2048": QwenCache}


def run_native(args, world, rank, local, pg):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rotated_lloyd_max_gb300 import build as b
    b.build()
    import rotated_lloyd_max_gb300 as tq
    tq.load()
    wl = WORKLOADS[args.workload](dev, seed_offset=0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    # warm-up (also compiles nothing: the library is AOT) and graph capture of the attention calls
    for _ in range(max(args.warmup, 3)):
        wl.encode_k(); wl.encode_v(); wl.attention()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        wl.attention()
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):
        flush.zero_(); wl.encode_k(); wl.encode_v(); graph.replay()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    barrier(pg)
    torch.cuda.synchronize()
    for s in range(K):
        flush.zero_()                     # L2 flush, outside the timed events
        e = ev[s]
        e[0].record(stream)
        wl.encode_k()
        e[1].record(stream)
        wl.encode_v()
        e[2].record(stream)
        graph.replay()
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    t_step = [e[0].elapsed_time(e[3]) / 1e3 for e in ev]
    t_enc = [(e[0].elapsed_time(e[2])) / 1e3 for e in ev]
    t_attn = [e[2].elapsed_time(e[3]) / 1e3 for e in ev]
    total = sum(t_step)
    total_max = max_over_ranks(pg, total, dev)
    bytes_all = sum_over_ranks(pg, wl.step_bytes * K, dev)
    value = bytes_all / total_max / 1e9
    enc_launch = sum(t_enc) / (2 * K)            # average encode launch
    attn_region = sum(t_attn) / K
    enc_bytes_per_launch = (wl.enc_in + wl.enc_out) / 2
    hbm, peak_kind = peaks()
    enc_gbs = enc_bytes_per_launch / enc_launch / 1e9
    attn_gbs = wl.attn_bytes / attn_region / 1e9
    dominant = "tq_encode" if sum(t_enc) >= sum(t_attn) else "tq_decode_attn"
    if dominant == "tq_encode":
        achieved, traffic = enc_gbs, None
    else:
        achieved, traffic = attn_gbs, None
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
                   "q_heads": wl.Hq, "head_dim": wl.d, "ctx": wl.ctx, "k_bits": wl.cfg["kb"],
                   "v_bits": wl.cfg["vb"], "bf16_layers": wl.dense, "l2": "flushed (256 MiB write) before each step",
                   "step": "encode whole cache (2 launches) + per-layer tq_decode_attn (graph replay)",
                   "parallelism": f"replicas x{world}"},
        "breakdown": {
            "encode_mvec_s": round(wl.vectors_per_step / (sum(t_enc) / K) / 1e6, 1),
            "encode_gbs": round(enc_gbs, 1),
            "decode_attn_kv_gbs": round(attn_gbs, 1),
            "decode_attn_tok_s": round(wl.tokens_per_step / attn_region, 1),
            "decode_attn_us_per_step": round(attn_region * 1e6, 2),
            "encode_us_per_step": round(sum(t_enc) / K * 1e6, 2),
            "step_algorithmic_bytes": wl.step_bytes,
        },
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "per_launch_bytes": enc_bytes_per_launch if dominant == "tq_encode" else wl.attn_bytes},
        "gpu_launches": wl.launches_per_step * K,
    }
    if clk:
        line["clocks"] = clk
    if not args.no_e2e:
        line["e2e"] = e2e_leg(wl, dev, graph, max(3, min(50, K)))
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        hin = wl.host_inputs()
        nbytes, secs = oracle_step(wl, hin)
        import oracle
        line["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s",
                                "cores": oracle.threads(), "kind": "oracle",
                                "sample": "one full step (all 28 layers: encode of the 22 compressed layers "
                                          "+ attention of every layer), fp64 C oracle"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_leg(wl, dev, graph, steps: int):
    """Same step through the public API with host buffers: pinned host inputs
    copied in, the step, the output copied back, all inside the timed region."""
    import torch
    pin = {k: t.cpu().pin_memory() for k, t in
           (("k_src", wl.k_src), ("v_src", wl.v_src), ("k_dense", wl.k_dense), ("v_dense", wl.v_dense),
            ("q", wl.q))}
    out_h = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()
    dst = {"k_src": wl.k_src, "v_src": wl.v_src, "k_dense": wl.k_dense, "v_dense": wl.v_dense, "q": wl.q}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = out_h.numel() * out_h.element_size()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        for k, t in pin.items():
            dst[k].copy_(t, non_blocking=True)
        wl.encode_k(); wl.encode_v(); graph.replay()
        out_h.copy_(wl.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    secs = (time.perf_counter() - t0) / steps
    return {"value": round(wl.step_bytes / secs / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3, 4)}


def run_reference(args, world, rank, local, pg):
    """The oracle (fp64 C, OpenMP) on the host cores: each step attends one
    (layer, kv head) unit of a compressed layer and one of a bf16 layer and
    encodes that unit's K/V, so K steps finish within minutes."""
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    import synth
    oracle.build()
    cfg = synth.CONFIGS[args.workload]
    d, ctx, Hkv, Hq = cfg["d"], cfg["ctx"], cfg["Hkv"], cfg["Hq"]
    G = Hq // Hkv
    okc = oracle.Codec(d=d, bits=cfg["kb"], seed=cfg["sign_seed"])
    ovc = oracle.Codec(d=d, bits=cfg["vb"], seed=cfg["sign_seed"])
    k = synth.gaussian_bf16((ctx, d), synth.layer_seed(cfg["data_seed"], 3, 0), fixed_channels=0)
    v = synth.gaussian_bf16((ctx, d), synth.layer_seed(cfg["data_seed"], 3, 1))
    kd = synth.gaussian_bf16((ctx, d), synth.layer_seed(cfg["data_seed"], 0, 0))
    vd = synth.gaussian_bf16((ctx, d), synth.layer_seed(cfg["data_seed"], 0, 1))
    q = synth.gaussian_bf16((G, d), synth.layer_seed(cfg["data_seed"], 3, 2), scale=cfg["q_scale"])

    def step():
        kr = oracle.encode_records(k, okc)
        vr = oracle.encode_records(v, ovc)
        oracle.unit_attention(q, okc, ovc, kr, vr, ctx, None, None, 1.0)
        oracle.unit_attention(q, None, None, None, None, 0, kd, vd, 1.0)
        return 2 * ctx * d * 2 + 2 * (kr.nbytes + vr.nbytes) + 2 * ctx * d * 2 + 2 * G * d * 6

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
        "config": {"workload": args.workload, "sample": "per step: encode one (layer, kv head) unit's K/V "
                   f"({ctx} tokens each) and attend it, plus one bf16-layer unit", "steps_run": n_run},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{n_run} steps of one compressed + one bf16 (layer, kv head) unit"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local, pg = dist_init(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, local, pg)
        else:
            run_native(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    main()
