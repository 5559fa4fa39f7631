"""Helpers shared by the tests: record unpacking (numpy, written from the
record format in include/tq.h), parity accounting against the oracle, and
device/host conversions.  Neither the CUDA path nor the oracle is imported
here; tests pass arrays in."""
from __future__ import annotations

import math

import numpy as np

CHUNK = 128


def record_layout(d: int, bits: int, outl: bool, cap: int):
    codes = CHUNK * d * bits // 8
    on, oc = codes, codes + 4 * CHUNK
    oe = oc + CHUNK
    return dict(norm=on, count=oc, entries=oe, size=(oe + 4 * cap) if outl else oc)


def unpack_records(rec: np.ndarray, n: int, d: int, bits: int, outl: bool = False, cap: int = 0):
    """Codes [n, d], norms [n] and per-token outlier dicts {idx: bf16 bits} of tokens 0..n-1."""
    lay = record_layout(d, bits, outl, cap)
    rec = np.ascontiguousarray(rec, np.uint8).reshape(-1, lay["size"])
    nrec = (n + CHUNK - 1) // CHUNK
    rb = d * bits // 8
    rows = rec[:nrec, :CHUNK * rb].reshape(nrec * CHUNK, rb)[:n]
    bitsarr = np.unpackbits(rows, axis=1, bitorder="little")[:, : d * bits].reshape(n, d, bits)
    codes = (bitsarr.astype(np.uint16) << np.arange(bits, dtype=np.uint16)).sum(-1).astype(np.uint8)
    norms = rec[:nrec, lay["norm"]:lay["norm"] + 4 * CHUNK].copy().view(np.float32).reshape(-1)[:n]
    outs = None
    if outl:
        outs = []
        for r in range(nrec):
            cnt = rec[r, lay["count"]:lay["count"] + CHUNK].astype(int)
            ent = rec[r, lay["entries"]:lay["entries"] + 4 * cap].copy().view(np.uint16).reshape(cap, 2)
            e = 0
            for i in range(min(CHUNK, n - r * CHUNK)):
                outs.append({int(ent[e + k, 0]): int(ent[e + k, 1]) for k in range(cnt[i])})
                e += cnt[i]
    return codes, norms, outs


def band_mask(y: np.ndarray, t32: np.ndarray, d: int, rel: float = 1e-6) -> np.ndarray:
    """Coordinates whose exact rotated value lies within `rel` (relative to the
    boundary, or to the coordinate scale 1/sqrt(d) for boundaries nearer zero)
    of a decision boundary."""
    t = t32.astype(np.float64)
    tol = rel * np.maximum(np.abs(t), 1.0 / math.sqrt(d))
    return np.any(np.abs(y[..., None] - t) <= tol, axis=-1)


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def check_codes(gpu_codes, enc, t32, d, total_frac=1e-5):
    """Codes equal except at band coordinates; returns (mismatches, band-size).
    With total_frac=None the caller aggregates the mismatch count over a whole
    workload (the bar is 1e-5 of all coordinates, not of one record)."""
    mism = gpu_codes != enc["codes"]
    band = band_mask(enc["y"], t32, d)
    outside = mism & ~band
    assert not outside.any(), (
        f"{int(outside.sum())} code mismatches outside the boundary band, first at "
        f"{tuple(int(v[0]) for v in np.nonzero(outside))}")
    if total_frac is not None:
        assert mism.sum() <= max(1, total_frac * mism.size), f"{int(mism.sum())} boundary mismatches"
    return int(mism.sum()), int(band.sum())


class MismatchTally:
    """Band differences over a workload -- boundary-band code mismatches plus
    outlier-list differences at the threshold or a bf16 rounding midpoint:
    at most 1e-5 of all coordinates."""

    def __init__(self):
        self.mism = 0
        self.total = 0

    def add(self, gpu_codes, enc, t32, d):
        m, _ = check_codes(gpu_codes, enc, t32, d, total_frac=None)
        self.mism += m
        self.total += gpu_codes.size

    def add_outliers(self, gpu_outs, enc, d, T):
        self.mism += check_outliers(gpu_outs, enc, d, T)

    def check(self, frac=1e-5):
        assert self.mism <= max(1, frac * self.total), f"{self.mism} band differences in {self.total} codes"


def check_norms(gpu_norms, enc, max_ulp=2):
    u = ulp_diff_f32(gpu_norms, enc["norms"])
    assert u.max() <= max_ulp, f"norm differs by {int(u.max())} ulp"
    return int(u.max())


def bf16_midpoint_band(y, rel: float = 1e-6):
    """True where the exact value y lies within `rel` (relative to |y|) of the
    midpoint between two consecutive bf16 values: there an f32 intermediate
    may round to either neighbour."""
    a = np.abs(np.asarray(y, np.float64))
    m, e = np.frexp(a)                                 # a = m * 2^e, 0.5 <= m < 1
    mid = (np.floor(m * 256.0) + 0.5) / 256.0 * np.exp2(e.astype(np.float64))
    return (a > 0) & (np.abs(a - mid) <= rel * a)


def check_outliers(gpu_outs, enc, d, T, rel=1e-6) -> int:
    """Outlier side lists against the oracle.  The stored set may differ only
    at coordinates whose exact |y| lies within `rel` of the threshold T/sqrt(d);
    a stored bf16 value may differ only by one bf16 step, and only where the
    exact y lies within `rel` of a bf16 rounding midpoint.  Every other
    difference fails.  Returns the number of band differences (set + value),
    which callers count with the boundary code mismatches."""
    thr = T / math.sqrt(d)
    y = enc["y"]
    n_band = 0
    for i, go in enumerate(gpu_outs):
        want = {int(j): int(enc["oval"][i, j]) for j in np.nonzero(enc["is_out"][i])[0]}
        for j in set(go) ^ set(want):
            assert abs(abs(y[i, j]) - thr) <= rel * thr, f"token {i} coord {j}: outlier set differs"
            n_band += 1
        for j in set(go) & set(want):
            if go[j] == want[j]:
                continue
            assert abs(int(go[j]) - int(want[j])) == 1 and bf16_midpoint_band(y[i, j], rel), (
                f"token {i} coord {j}: outlier value {go[j]:#06x} != {want[j]:#06x} (y = {y[i, j]!r})")
            n_band += 1
    return n_band


def to_bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_tensor_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
