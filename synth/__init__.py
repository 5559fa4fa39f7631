"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds input generation only -- random draws and bf16 rounding of
them -- and none of the codec's or the attention's arithmetic.  It is the one
module both the CUDA path's callers and the oracle's callers use, so that both
sides see identical inputs.

Two back ends:
  * numpy (PCG64) on the host, for small cases the oracle finishes quickly;
  * torch generators on the device, for full-size caches (tens of GB) where host
    generation would dominate; the oracle then receives host copies of sampled
    slices of the very same tensors.

Distributions follow the workloads the pages describe (see the recipe table in
the design notes): N(0,1) entries, per-vector LogNormal scales, fixed
channels scaled x8, 2% N(0,36) outlier coordinates, and q ~ N(0,1)/sqrt(d).
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# bf16 rounding of generated data (input preparation, round to nearest even)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Host generators (numpy)
# ---------------------------------------------------------------------------


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def gaussian_bf16(shape, seed: int, lognormal_sigma: float | None = None,
                  fixed_channels: int = 0, channel_scale: float = 8.0,
                  outlier_frac: float = 0.0, outlier_std: float = 6.0,
                  scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0,1) rows (last axis = head_dim), optionally:
      * times a per-row LogNormal(0, sigma) scale,
      * with `fixed_channels` channels per leading-index group scaled x channel_scale
        (the same channels for every row of a group: shape[:-2] indexes groups),
      * with a fraction of coordinates drawn from N(0, outlier_std^2) instead,
      * times a constant `scale`."""
    g = rng(seed)
    shape = tuple(shape)
    x = g.standard_normal(shape, dtype=np.float32)
    if outlier_frac > 0.0:
        m = g.random(shape, dtype=np.float32) < outlier_frac
        x = np.where(m, outlier_std * g.standard_normal(shape, dtype=np.float32), x)
    if lognormal_sigma is not None:
        s = np.exp(lognormal_sigma * g.standard_normal(shape[:-1] + (1,), dtype=np.float32))
        x = x * s.astype(np.float32)
    if fixed_channels:
        d = shape[-1]
        groups = shape[:-2] if len(shape) > 2 else ()
        mult = np.ones(groups + (1, d), np.float32)
        for idx in np.ndindex(*groups) if groups else [()]:
            ch = g.choice(d, size=fixed_channels, replace=False)
            mult[idx + (0,)][ch] = channel_scale
        x = x * mult
    return f32_to_bf16_bits((x * np.float32(scale)).astype(np.float32))


# ---------------------------------------------------------------------------
# Device generators (torch)
# ---------------------------------------------------------------------------


def torch_gaussian_bf16(shape, seed: int, device, lognormal_sigma: float | None = None,
                        fixed_channels: int = 0, channel_scale: float = 8.0,
                        outlier_frac: float = 0.0, outlier_std: float = 6.0,
                        scale: float = 1.0, out=None):
    """Same recipe as `gaussian_bf16`, drawn by a torch generator on `device`
    (its stream differs from numpy's; sizes here are the full workloads).
    Returns a bf16 tensor (or fills `out`)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = tuple(shape)
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_frac > 0.0:
        m = torch.rand(shape, generator=gen, device=device) < outlier_frac
        x = torch.where(m, outlier_std * torch.randn(shape, generator=gen, device=device), x)
        del m
    if lognormal_sigma is not None:
        x *= torch.exp(lognormal_sigma * torch.randn(shape[:-1] + (1,), generator=gen,
                                                    device=device))
    if fixed_channels:
        d = shape[-1]
        groups = shape[:-2] if len(shape) > 2 else ()
        n_groups = int(np.prod(groups)) if groups else 1
        keys = torch.rand((n_groups, d), generator=gen, device=device)
        ch = keys.argsort(dim=1)[:, :fixed_channels]
        mult = torch.ones((n_groups, d), device=device)
        mult.scatter_(1, ch, channel_scale)
        x = (x.reshape((n_groups, -1, d)) * mult[:, None, :]).reshape(shape)
    if scale != 1.0:
        x *= scale
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


# ---------------------------------------------------------------------------
# Workload recipes (shapes and distributions of the five configurations)
# ---------------------------------------------------------------------------

CONFIGS = {
    # codec round trip, no attention
    "codec_roundtrip_4096x128_b3": dict(
        kind="codec", n=4096, d=128, bits=3, sign_seed=1, data_seed=0, lognormal_sigma=0.5),
    # Qwen2-1.5B-shaped cache (DS-Distill geometry)
    "qwen2_1p5b_ctx2048": dict(
        kind="attn", L=28, B=1, Hkv=2, Hq=12, d=128, ctx=2048, kb=3, vb=2,
        dense_layers=(0, 1, 2, 25, 26, 27), tail=0, k_fixed_channels=4, q_scale=1 / math.sqrt(128),
        T=0.0, shared_kv=False, data_seed=0, sign_seed=1),
    # DeepSeek-V4-Flash-like MQA
    "v4flash_mqa_ctx65536": dict(
        kind="attn", L=43, B=1, Hkv=1, Hq=64, d=512, ctx=65536, kb=4, vb=4,
        dense_layers=(), window=128, margin=16, t_q=1, tail=256, k_lognormal_sigma=0.3,
        q_scale=1 / math.sqrt(512), T=0.0, shared_kv=True, data_seed=0, sign_seed=1),
    # batched decode over a compressed cache with outliers
    "batched_b32_ctx32768": dict(
        kind="attn", L=32, B=32, Hkv=8, Hq=32, d=128, ctx=32768, kb=4, vb=3,
        dense_layers=(), tail=0, k_outlier_frac=0.02, q_scale=1 / math.sqrt(128), T=2.0,
        shared_kv=False, data_seed=0, sign_seed=1),
    # long context
    "longctx_b4_ctx262144": dict(
        kind="attn", L=8, B=4, Hkv=8, Hq=32, d=128, ctx=262144, kb=3, vb=2,
        dense_layers=(), tail=1024, q_scale=1 / math.sqrt(128), T=0.0, shared_kv=False,
        data_seed=0, sign_seed=1),
    # encode sweep
    "encode_sweep_16M": dict(kind="sweep", n=1 << 24, ds=(64, 128, 256, 512), bits=(2, 3, 4),
                             data_seed=0, sign_seed=1),
}


def layer_seed(data_seed: int, layer: int, stream: int) -> int:
    """Seed of one layer's K (stream 0), V (stream 1) or q (stream 2) draw."""
    return data_seed * 1_000_003 + layer * 16 + stream


def kv_recipe(cfg: dict, stream: str) -> dict:
    """Distribution keywords of the K or V draw of an attention config."""
    kw = {}
    if stream == "k":
        if cfg.get("k_fixed_channels"):
            kw["fixed_channels"] = cfg["k_fixed_channels"]
        if cfg.get("k_lognormal_sigma") is not None:
            kw["lognormal_sigma"] = cfg["k_lognormal_sigma"]
        if cfg.get("k_outlier_frac"):
            kw["outlier_frac"] = cfg["k_outlier_frac"]
    return kw
