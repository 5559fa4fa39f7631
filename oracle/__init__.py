"""CPU oracle for the rotated Lloyd-Max KV-cache codec and its decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` import this package.  It shares no code with
the CUDA path (``rotated_lloyd_max_gb300``) and never imports it.

The arithmetic lives in ``tq_oracle.c`` (plain C, fp64, built by ``build()``
with ``-ffp-contract=off`` so that x86 and Arm hosts round identically); this
module only marshals numpy arrays and composes the C steps in the order the
method states them.  See the header of ``tq_oracle.c`` for the sources and the
readings taken where the pages are silent.

Parity unpinned: the sign generator (SplitMix64) and the record bit order are
this project's own definitions; they are pinned by hand-worked examples and the
published SplitMix64 vectors, not by the pages.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
CHUNK = 128

_lib = None


def build(force: bool = False) -> str:
    """Compile tq_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint64
        sig = {
            "orc_lloyd_max_gaussian": (i32, [i32, P, P, P]),
            "orc_codebook_f32": (None, [i32, i32, P, P]),
            "orc_splitmix64_next": (u64, [P]),
            "orc_signs": (None, [u64, i32, P]),
            "orc_fwht": (None, [P, i32]),
            "orc_bf16_to_double": (f64, [ctypes.c_uint16]),
            "orc_double_to_bf16": (ctypes.c_uint16, [f64]),
            "orc_record_layout": (i64, [i32, i32, i32, i32, P, P, P]),
            "orc_encode_vectors": (None, [P, i64, i32, i64, i32, P, P, P, f64, i32, P, P, P, P, P]),
            "orc_midpoints_f32": (None, [i32, P, P]),
            "orc_pack_record": (None, [i32, i32, i32, i32, i32, P, P, P, P, P]),
            "orc_read_code": (i32, [P, i32, i32]),
            "orc_decode_records": (None, [P, i64, i64, i32, i32, i32, i32, P, P, i32, P]),
            "orc_attention": (None, [P, i32, P, P, i64, i32, f64, f64, P]),
            "orc_attention_rotated": (None, [P, i32, P, P, i64, P, P, i64, i32, f64, f64, P, P, P]),
            "orc_retention_floor": (i32, [i32, i32, i32]),
            "orc_chunks_to_evict": (i32, [i32, i32, i32, i32, i32]),
            "orc_bf16_round_array": (None, [P, i64, P]),
            "orc_attention_sparse_v": (None, [P, i32, P, P, i64, i32, f64, f64, f64, i32, P, P, P, i32, i32, P,
                                              P]),
            "orc_rollback_counts": (i32, [i32, i32, i32, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


# ---------------------------------------------------------------------------
# Codebook and signs
# ---------------------------------------------------------------------------
def lloyd_max_gaussian(bits: int):
    """(centroids, boundaries, mse, iterations) of the unit-variance table."""
    K = 1 << bits
    c = np.zeros(K, np.float64)
    t = np.zeros(max(K - 1, 1), np.float64)
    mse = np.zeros(1, np.float64)
    it = _load().orc_lloyd_max_gaussian(bits, _p(c), _p(t), _p(mse))
    return c, t[:K - 1], float(mse[0]), it


def codebook_f32(bits: int, d: int):
    """f32 centroids (scaled by 1/sqrt(d)) and their f32 midpoints."""
    K = 1 << bits
    c = np.zeros(K, np.float32)
    t = np.zeros(max(K - 1, 1), np.float32)
    _load().orc_codebook_f32(bits, d, _p(c), _p(t))
    return c, t[:K - 1]


def midpoints_f32(bits: int, c32: np.ndarray) -> np.ndarray:
    """f32 midpoints of an ascending f32 centroid table (its decision boundaries)."""
    c = np.ascontiguousarray(c32, np.float32)
    t = np.zeros(max((1 << bits) - 1, 1), np.float32)
    _load().orc_midpoints_f32(bits, _p(c), _p(t))
    return t[:(1 << bits) - 1]


def splitmix64(seed: int, n: int) -> np.ndarray:
    st = (ctypes.c_uint64 * 1)(seed)
    lib = _load()
    return np.array([lib.orc_splitmix64_next(ctypes.cast(st, ctypes.c_void_p)) for _ in range(n)],
                    dtype=np.uint64)


def signs(seed: int, d: int) -> np.ndarray:
    s = np.zeros(d, np.int8)
    _load().orc_signs(seed, d, _p(s))
    return s


def fwht(v: np.ndarray) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform of each row (fp64)."""
    out = np.array(v, dtype=np.float64, copy=True, order="C")
    lib = _load()
    rows = out.reshape(-1, out.shape[-1])
    for r in rows:
        lib.orc_fwht(_p(r), r.shape[0])
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    u = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16(y: float) -> int:
    return int(_load().orc_double_to_bf16(float(y)))


# ---------------------------------------------------------------------------
# Codec
# ---------------------------------------------------------------------------
def default_outlier_cap(d: int) -> int:
    """Entries per 128-token record: 8% of the record's coordinates, rounded up
    to a multiple of 4 (the 8% slot sizing of "v1.3 PPL on vLLM: production cell +
    per-channel attribution", M6 Phase A, is the precedent)."""
    return 4 * ((8 * CHUNK * d + 399) // 400)


SCALE_MODES = {"norm": 0, "matched_norm": 1, "inner_product": 2, "least_squares": 3}


@dataclass(frozen=True)
class Codec:
    d: int
    bits: int
    seed: int = 1
    T: float = 0.0          # 0: no outlier section
    cap: int = 0            # entries per record (0: default)
    centroids: tuple = ()   # caller-supplied ascending f32 table (2^bits values); () = the Gaussian table
    scale: str = "norm"     # stored per-vector scale (see orc_encode_vector)

    @property
    def has_outliers(self) -> bool:
        return self.T != 0.0

    @property
    def outlier_cap(self) -> int:
        return self.cap or default_outlier_cap(self.d)

    @property
    def row_bytes(self) -> int:
        return self.d * self.bits // 8

    def layout(self):
        on, oc, oe = (ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64())
        size = _load().orc_record_layout(self.d, self.bits, int(self.has_outliers), self.outlier_cap,
                                         ctypes.byref(on), ctypes.byref(oc), ctypes.byref(oe))
        return dict(size=size, norm=on.value, count=oc.value, entries=oe.value)

    @property
    def record_bytes(self) -> int:
        return self.layout()["size"]

    def tables(self):
        if self.centroids:
            c = np.array(self.centroids, np.float32)
            assert c.shape == (1 << self.bits,)
            t = midpoints_f32(self.bits, c)
        else:
            c, t = codebook_f32(self.bits, self.d)
        return c, t, signs(self.seed, self.d)


def encode_vectors(x_bf16: np.ndarray, codec: Codec, want_y: bool = False):
    """Per-vector encode of rows of bf16 bit patterns [n, d] (uint16).

    Returns dict(codes [n,d] u8, norms [n] f32, is_out [n,d] u8, oval [n,d] u16, y [n,d] f64)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n, d = x.shape
    assert d == codec.d
    c, t, s = codec.tables()
    codes = np.zeros((n, d), np.uint8)
    norms = np.zeros(n, np.float32)
    is_out = np.zeros((n, d), np.uint8)
    oval = np.zeros((n, d), np.uint16)
    y = np.zeros((n, d), np.float64) if want_y else None
    T = codec.T if codec.has_outliers else 0.0
    _load().orc_encode_vectors(_p(x), n, d, d, codec.bits, _p(np.ascontiguousarray(c)),
                               _p(np.ascontiguousarray(t)), _p(s), T, SCALE_MODES[codec.scale],
                               _p(codes), _p(norms), _p(is_out), _p(oval),
                               _p(y) if y is not None else None)
    return dict(codes=codes, norms=norms, is_out=is_out, oval=oval, y=y)


def pack_records(enc: dict, codec: Codec, n_records: int | None = None) -> np.ndarray:
    """Pack per-vector encodings of tokens 0..n-1 into records [n_rec, bytes]."""
    n = enc["codes"].shape[0]
    nrec = n_records if n_records is not None else (n + CHUNK - 1) // CHUNK
    rec = np.zeros((nrec, codec.record_bytes), np.uint8)
    lib = _load()
    for r in range((n + CHUNK - 1) // CHUNK):
        a, b = r * CHUNK, min(n, (r + 1) * CHUNK)
        sl = lambda k: np.ascontiguousarray(enc[k][a:b])
        lib.orc_pack_record(codec.d, codec.bits, int(codec.has_outliers), codec.outlier_cap, b - a,
                            _p(sl("codes")), _p(sl("norms")), _p(sl("is_out")), _p(sl("oval")),
                            _p(rec[r]))
    return rec


def encode_records(x_bf16: np.ndarray, codec: Codec) -> np.ndarray:
    return pack_records(encode_vectors(x_bf16, codec), codec)


def read_code(row: np.ndarray, j: int, bits: int) -> int:
    return int(_load().orc_read_code(_p(np.ascontiguousarray(row, np.uint8)), j, bits))


def decode_records(records: np.ndarray, n: int, codec: Codec, rotated: bool = False) -> np.ndarray:
    """Decode tokens [0, n) of a record array -> fp64 [n, d] (original basis,
    or n_i * yhat_i in the rotated basis when ``rotated``)."""
    rec = np.ascontiguousarray(records, np.uint8).reshape(-1, codec.record_bytes)
    c, _, s = codec.tables()
    out = np.zeros((n, codec.d), np.float64)
    if n:
        _load().orc_decode_records(_p(rec), codec.record_bytes, n, codec.d, codec.bits,
                                   int(codec.has_outliers), codec.outlier_cap, _p(c), _p(s),
                                   int(rotated), _p(out))
    return out


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, softcap: float = 0.0) -> np.ndarray:
    """Brute-force softmax attention in fp64.  q [G, d], K/V [n, d] -> [G, d].
    softcap > 0 caps each logit s = scale * q.k to softcap * tanh(s / softcap)."""
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    G, d = q.shape
    out = np.zeros((G, d), np.float64)
    _load().orc_attention(_p(q), G, _p(K), _p(V), K.shape[0], d, float(scale), float(softcap), _p(out))
    return out


def attention_sparse_v(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, eps: float, group: int,
                       blocks, softcap: float = 0.0):
    """Attention with sparse-V skipping (see orc_attention_sparse_v) in fp64.
    blocks: list of (begin, end, sequence) token ranges, each sequence's
    blocks in visiting order.  Returns (out [G, d], skipped (group, token) pairs)."""
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    G, d = q.shape
    bb = np.ascontiguousarray([b[0] for b in blocks] or [0], np.int64)
    be = np.ascontiguousarray([b[1] for b in blocks] or [0], np.int64)
    bs = np.ascontiguousarray([b[2] for b in blocks] or [0], np.int32)
    n_seq = (max(b[2] for b in blocks) + 1) if blocks else 0
    out = np.zeros((G, d), np.float64)
    sk = np.zeros(1, np.int64)
    _load().orc_attention_sparse_v(_p(q), G, _p(K), _p(V), K.shape[0], d, float(scale), float(softcap),
                                   float(eps), int(group), _p(bb), _p(be), _p(bs), len(blocks), n_seq, _p(out),
                                   _p(sk))
    return out, int(sk[0])


def sparse_v_blocks(n_records: int, records_per_split: int, warps: int = 4, groups: int = 1):
    """The blocks of the tensor-core decode kernel's schedule: split s covers
    records [s cps, (s+1) cps); a CTA of `groups` 4-warp groups deals them out
    round robin (group g takes records s cps + g, s cps + g + groups, ...);
    within a group, warp w visits the tokens [128 r + 32 w, 128 r + 32 w + 32)
    of its records in order, sharing one running maximum (a sequence per
    (split, group, warp))."""
    blocks = []
    span = 128 // warps
    n_split = (n_records + records_per_split - 1) // records_per_split if n_records else 0
    for s_ in range(n_split):
        end = min((s_ + 1) * records_per_split, n_records)
        for g in range(groups):
            for w in range(warps):
                for r in range(s_ * records_per_split + g, end, groups):
                    blocks.append((128 * r + span * w, 128 * r + span * (w + 1), (s_ * groups + g) * warps + w))
    return blocks


def unit_attention_sparse_v(q_bf16, codec_k: Codec, codec_v: Codec, k_rec, v_rec, n_comp, k_dense_bf16,
                            v_dense_bf16, scale, eps, records_per_split, heads_per_cta, softcap=0.0, groups=1):
    """unit_attention with sparse-V skipping over the compressed tokens, on the
    tensor-core kernel's schedule (sparse_v_blocks); dense tokens are never
    skipped.  Returns (out, skipped (group, token) pairs)."""
    q = bf16_to_f64(q_bf16)
    d = q.shape[1]
    Ks, Vs = [decode_records(k_rec, n_comp, codec_k)], [decode_records(v_rec, n_comp, codec_v)]
    if k_dense_bf16 is not None and len(k_dense_bf16):
        Ks.append(bf16_to_f64(k_dense_bf16).reshape(-1, d))
        Vs.append(bf16_to_f64(v_dense_bf16).reshape(-1, d))
    blocks = sparse_v_blocks(n_comp // 128, records_per_split, groups=groups)
    return attention_sparse_v(q, np.concatenate(Ks), np.concatenate(Vs), scale, eps, heads_per_cta, blocks, softcap)


def attention_rotated(q, Kr, Vr, Kd, Vd, scale, sk, sv, softcap=0.0):
    """Rotated-domain evaluation of the same attention (cross-check only)."""
    q = np.ascontiguousarray(q, np.float64)
    G, d = q.shape
    f = lambda a: np.ascontiguousarray(a, np.float64).reshape(-1, d)
    Kr, Vr, Kd, Vd = f(Kr), f(Vr), f(Kd), f(Vd)
    out = np.zeros((G, d), np.float64)
    _load().orc_attention_rotated(_p(q), G, _p(Kr), _p(Vr), Kr.shape[0], _p(Kd), _p(Vd),
                                  Kd.shape[0], d, float(scale), float(softcap),
                                  _p(np.ascontiguousarray(sk, np.int8)),
                                  _p(np.ascontiguousarray(sv, np.int8)), _p(out))
    return out


def unit_attention(q_bf16, codec_k: Codec | None, codec_v: Codec | None, k_rec, v_rec, n_comp,
                   k_dense_bf16, v_dense_bf16, scale, softcap=0.0):
    """Decode-attention output for one (layer, batch, kv-head) unit.

    q_bf16 [G, d] uint16; compressed tokens 0..n_comp-1 in k_rec/v_rec (records);
    dense tokens (bf16 [nd, d] uint16, any order) from the tail or a bf16 layer.
    Keys/values are fully dequantised to the original basis and attended by
    brute force in fp64."""
    q = bf16_to_f64(q_bf16)
    d = q.shape[1]
    Ks, Vs = [], []
    if n_comp:
        Ks.append(decode_records(k_rec, n_comp, codec_k))
        Vs.append(decode_records(v_rec, n_comp, codec_v))
    if k_dense_bf16 is not None and len(k_dense_bf16):
        Ks.append(bf16_to_f64(k_dense_bf16).reshape(-1, d))
        Vs.append(bf16_to_f64(v_dense_bf16).reshape(-1, d))
    K = np.concatenate(Ks) if Ks else np.zeros((0, d))
    V = np.concatenate(Vs) if Vs else np.zeros((0, d))
    return attention(q, K, V, scale, softcap)


# ---------------------------------------------------------------------------
# Chunked eviction
# ---------------------------------------------------------------------------
def retention_floor(window: int, t_q: int, margin: int) -> int:
    return int(_load().orc_retention_floor(window, t_q, margin))


def chunks_to_evict(tail_len: int, window: int, t_q: int, margin: int, chunk: int = CHUNK) -> int:
    return int(_load().orc_chunks_to_evict(tail_len, window, t_q, margin, chunk))


def evict(tail_k, tail_v, start: int, length: int, n_chunks: int, k_rec, v_rec, codec_k: Codec,
          codec_v: Codec | None, window: int, t_q: int, margin: int):
    """Chunked eviction of one (layer, batch) unit, every kv head.

    tail_k/tail_v: bf16 ring buffers [Hkv, cap, d] (uint16); k_rec/v_rec: record
    arrays [Hkv, rec_cap, bytes] (modified in place; v_rec None when keys and
    values share records).  The oldest whole chunks beyond the retention floor
    are encoded into records n_chunks, n_chunks+1, ... and the counters advance.
    Returns (start, length, n_chunks)."""
    cap = tail_k.shape[1]
    k = chunks_to_evict(length, window, t_q, margin)
    for e in range(k):
        slots = (start + e * CHUNK + np.arange(CHUNK)) % cap
        for h in range(tail_k.shape[0]):
            k_rec[h, n_chunks + e] = encode_records(tail_k[h, slots], codec_k)[0]
            if v_rec is not None:
                v_rec[h, n_chunks + e] = encode_records(tail_v[h, slots], codec_v)[0]
    return (start + k * CHUNK) % cap, length - k * CHUNK, n_chunks + k


# ---------------------------------------------------------------------------
# Rollback
# ---------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """bf16 bits (nearest, ties to even) of every value of a fp64 array."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros(x.shape, np.uint16)
    _load().orc_bf16_round_array(_p(x), x.size, _p(out))
    return out


def rollback_counts(n_chunks: int, tail_len: int, new_len: int):
    """(n_chunks', tail_len', start reset?, tokens to decode) of a rollback."""
    n, ln, rs = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    m = _load().orc_rollback_counts(n_chunks, tail_len, new_len, ctypes.byref(n), ctypes.byref(ln),
                                    ctypes.byref(rs))
    return n.value, ln.value, bool(rs.value), m


def rollback(tail_k, tail_v, start: int, length: int, n_chunks: int, k_rec, v_rec, codec_k: Codec,
             codec_v: Codec | None, new_len: int):
    """Rollback of one (layer, batch) unit, every kv head (see orc_rollback_counts).

    tail_k/tail_v: bf16 ring buffers [Hkv, cap, d] (uint16, modified in place;
    tail_v None when keys and values share records and ring); k_rec/v_rec:
    record arrays [Hkv, rec_cap, bytes] (read only).  On a deep rollback the m
    remaining tokens of record n' are decoded (fp64) and rounded to bf16 into
    ring slots 0..m-1.  Returns (start, length, n_chunks)."""
    n2, len2, reset, m = rollback_counts(n_chunks, length, new_len)
    if not reset:
        return start, len2, n2
    for h in range(tail_k.shape[0]):
        for tail, rec, cod in ((tail_k, k_rec, codec_k), (tail_v, v_rec, codec_v)):
            if tail is None or m == 0:
                continue
            x = decode_records(rec[h, n2:n2 + 1], m, cod)
            tail[h, :m] = bf16_round(x)
    return 0, len2, n2

