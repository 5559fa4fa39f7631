"""Python binding of libtq_gb300 (the sm_103a rotated Lloyd-Max KV-cache codec
and fused decode attention).

Argument marshalling only: every step of the codec and the attention runs in
the library's CUDA kernels.  Torch tensors supply device memory and the
current CUDA stream.  The functions carry the C names of ``include/tq.h``.
There is no CPU fallback: if the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq_gb300.so")
CHUNK = 128

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA = range(5)

c_i32, c_i64, c_u64, c_f32, c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p


class tq_codec(ctypes.Structure):
    _fields_ = [("head_dim", c_i32), ("bits", c_i32), ("sign_seed", c_u64), ("outlier_T", c_f32),
                ("outlier_cap", c_i32), ("centroids", c_f32 * 16), ("boundaries", c_f32 * 15),
                ("sign_bits", ctypes.c_uint32 * 16), ("scale_mode", c_i32)]


class tq_evict_args(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("batch", c_i32), ("n_kv_heads", c_i32),
                ("k_rec", c_p), ("v_rec", c_p), ("k_rec_layer_stride", c_i64),
                ("v_rec_layer_stride", c_i64), ("rec_cap", c_i32),
                ("k_tail", c_p), ("v_tail", c_p), ("tail_layer_stride", c_i64), ("tail_cap", c_i32),
                ("n_chunks", c_p), ("tail_start", c_p), ("tail_len", c_p),
                ("window", c_i32), ("margin", c_i32), ("t_q", c_i32), ("max_evict", c_i32),
                ("block_table", c_p), ("table_stride", c_i32)]


class tq_attn_args(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("batch", c_i32), ("n_q_heads", c_i32), ("n_kv_heads", c_i32),
                ("head_dim", c_i32), ("scale", c_f32),
                ("q", c_p), ("q_layer_stride", c_i64), ("q_batch_stride", c_i64),
                ("out", c_p),
                ("k_rec", c_p), ("v_rec", c_p), ("k_rec_layer_stride", c_i64),
                ("v_rec_layer_stride", c_i64), ("rec_cap", c_i32),
                ("k_tail", c_p), ("v_tail", c_p), ("tail_layer_stride", c_i64), ("tail_cap", c_i32),
                ("n_chunks", c_p), ("tail_start", c_p), ("tail_len", c_p),
                ("max_chunks", c_i32), ("max_tail", c_i32), ("splits", c_i32), ("cuda_core_path", c_i32),
                ("softcap", c_f32), ("block_table", c_p), ("table_stride", c_i32), ("sparse_v_eps", c_f32)]


class tq_attn_plan(ctypes.Structure):
    _fields_ = [("compressed_kernel", c_i32), ("dense_kernel", c_i32), ("compressed_splits", c_i32),
                ("dense_splits", c_i32), ("records_per_split", c_i32), ("dense_tokens_per_split", c_i32),
                ("heads_per_cta", c_i32), ("dense_heads_per_cta", c_i32), ("launches", c_i32),
                ("warps_per_cta", c_i32), ("workspace_bytes", c_u64)]


ATTN_KERNELS = {0: "none", 1: "cuda_core", 2: "cuda_core_warp", 3: "mma", 4: "mma512", 5: "tcgen05"}

_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tq_version": (ctypes.c_int, []),
    "tq_codebook_scratch_bytes": (ctypes.c_size_t, []),
    "tq_make_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, c_u64, c_f32, ctypes.c_int, c_p,
                                        ctypes.c_size_t, ctypes.POINTER(tq_codec),
                                        ctypes.POINTER(ctypes.c_double), c_p]),
    "tq_record_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_codec)]),
    "tq_codec_set_centroids": (ctypes.c_int, [ctypes.POINTER(tq_codec), ctypes.POINTER(c_f32), ctypes.c_int]),
    "tq_encode": (ctypes.c_int, [ctypes.POINTER(tq_codec), c_p, c_i64, c_i64, c_i64, c_i64, c_p, c_i64,
                                 c_i64, c_p]),
    "tq_decode": (ctypes.c_int, [ctypes.POINTER(tq_codec), c_p, c_i64, c_i64, c_i64, c_i64, c_p, c_i64,
                                 c_i64, c_p]),
    "tq_evict": (ctypes.c_int, [ctypes.POINTER(tq_codec), ctypes.POINTER(tq_codec),
                                ctypes.POINTER(tq_evict_args), c_p]),
    "tq_rollback": (ctypes.c_int, [ctypes.POINTER(tq_codec), ctypes.POINTER(tq_codec),
                                   ctypes.POINTER(tq_evict_args), c_p, c_p]),
    "tq_decode_attn_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(tq_attn_args),
                                                        ctypes.POINTER(tq_codec),
                                                        ctypes.POINTER(tq_codec)]),
    "tq_decode_attn": (ctypes.c_int, [ctypes.POINTER(tq_attn_args), ctypes.POINTER(tq_codec),
                                      ctypes.POINTER(tq_codec), c_p, ctypes.c_size_t, c_p]),
    "tq_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(tq_attn_args), ctypes.POINTER(tq_codec),
                                              ctypes.POINTER(tq_codec), c_p]),
    "tq_decode_attn_plan": (ctypes.c_int, [ctypes.POINTER(tq_attn_args), ctypes.POINTER(tq_codec),
                                           ctypes.POINTER(tq_codec), ctypes.POINTER(tq_attn_plan)]),
}

NOALLOC_WORKSPACE_BYTES = 8 << 20

_lib = None


class TqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


def load(path: str | None = None):
    """Load libtq_gb300.so (built by ``rotated_lloyd_max_gb300.build``)."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with `python -m rotated_lloyd_max_gb300.build` "
                              "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().tq_status_string(status).decode()


def _check(fn: str, status: int):
    if status != TQ_OK:
        raise TqError(fn, status)


def _stream(stream):
    import torch
    if stream is None:
        return c_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return c_p(stream)
    return c_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else c_p(t.data_ptr())


# ---------------------------------------------------------------------------
# codec
# ---------------------------------------------------------------------------
@dataclass
class Codec:
    """A tq_codec filled by the device-side Lloyd-Max kernel."""
    c: tq_codec
    mse: float

    @property
    def head_dim(self):
        return self.c.head_dim

    @property
    def bits(self):
        return self.c.bits

    @property
    def record_bytes(self) -> int:
        return tq_record_bytes(self)

    def centroids(self):
        return list(self.c.centroids)[: 1 << self.c.bits]

    def boundaries(self):
        return list(self.c.boundaries)[: (1 << self.c.bits) - 1]

    def sign_words(self):
        return list(self.c.sign_bits)[: self.c.head_dim // 32]


def tq_make_codebook(bits: int, head_dim: int, sign_seed: int = 1, outlier_T: float = 0.0,
                     outlier_cap: int = 0, device=None, stream=None) -> Codec:
    import torch
    lib = load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    scratch = torch.empty(int(lib.tq_codebook_scratch_bytes()), dtype=torch.uint8, device=dev)
    out = tq_codec()
    mse = ctypes.c_double()
    _check("tq_make_codebook", lib.tq_make_codebook(bits, head_dim, sign_seed, float(outlier_T), outlier_cap,
                                                    _ptr(scratch), scratch.numel(), ctypes.byref(out),
                                                    ctypes.byref(mse), _stream(stream)))
    return Codec(out, mse.value)


SCALE_MODES = {"norm": 0, "matched_norm": 1, "inner_product": 2, "least_squares": 3}


def tq_codec_set_centroids(codec: Codec, centroids) -> Codec:
    """A copy of `codec` using the caller's ascending f32 table (2^bits values)."""
    vals = [float(v) for v in centroids]
    out = Codec(tq_codec.from_buffer_copy(codec.c), codec.mse)
    arr = (c_f32 * len(vals))(*vals)
    _check("tq_codec_set_centroids", load().tq_codec_set_centroids(ctypes.byref(out.c), arr, len(vals)))
    return out


def with_scale(codec: Codec, mode: str) -> Codec:
    """A copy of `codec` storing the per-vector scale `mode` (see SCALE_MODES)."""
    out = Codec(tq_codec.from_buffer_copy(codec.c), codec.mse)
    out.c.scale_mode = SCALE_MODES[mode]
    return out


def tq_record_bytes(codec: Codec) -> int:
    n = load().tq_record_bytes(ctypes.byref(codec.c))
    if n == 0:
        raise TqError("tq_record_bytes", TQ_ERR_INVALID_ARG)
    return int(n)


def _groups(t, inner: int):
    """(n_groups, n_rows, row_stride, group_stride) of a [.., rows, inner] view."""
    if t.dim() == 2:
        return 1, t.shape[0], t.stride(0), 0
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.stride(1), t.stride(0)
    raise ValueError("expected a 2-D [rows, inner] or 3-D [groups, rows, inner] tensor")


def tq_encode(codec: Codec, src, dst, first_vec: int = 0, stream=None):
    """Encode bf16 vectors src [n_vec, d] or [groups, n_vec, d] (last dim contiguous) into the
    record array dst (uint8 [n_rec, record_bytes] or [groups, n_rec, record_bytes])."""
    import torch
    assert src.dtype == torch.bfloat16 and src.stride(-1) == 1 and src.shape[-1] == codec.head_dim
    assert dst.dtype == torch.uint8 and dst.stride(-1) == 1
    g, n, vs, gs = _groups(src, codec.head_dim)
    dg = dst.stride(0) if dst.dim() == 3 else 0
    _check("tq_encode", load().tq_encode(ctypes.byref(codec.c), _ptr(src), g, n, vs, gs, _ptr(dst), dg,
                                         first_vec, _stream(stream)))


def tq_decode(codec: Codec, src, dst, first_vec: int = 0, stream=None):
    """Decode tokens [first_vec, first_vec + n) of record arrays src into f32 dst [.., n, d]."""
    import torch
    assert dst.dtype == torch.float32 and dst.stride(-1) == 1 and dst.shape[-1] == codec.head_dim
    assert src.dtype == torch.uint8
    g, n, vs, gs = _groups(dst, codec.head_dim)
    sg = src.stride(0) if src.dim() == 3 else 0
    _check("tq_decode", load().tq_decode(ctypes.byref(codec.c), _ptr(src), g, n, sg, first_vec, _ptr(dst),
                                         vs, gs, _stream(stream)))


def make_evict_args(*, k_rec, v_rec, k_tail, v_tail, n_chunks, tail_start, tail_len, window: int, margin: int,
                    t_q: int = 1, max_evict: int = 1, block_table=None) -> tq_evict_args:
    """tq_evict_args from tensors.  k_rec/v_rec: uint8 [L, B, Hkv, rec_cap, record_bytes]
    (v_rec may be k_rec for shared keys/values) or, with block_table (int32
    [B, table_stride]), per-layer pools uint8 [L, n_blocks, Hkv, record_bytes];
    k_tail/v_tail: bf16 [L, B, Hkv, tail_cap, d]; counters: int32 [L, B]."""
    if block_table is None:
        L, B, Hkv, rec_cap = k_rec.shape[:4]
        table, stride = None, 0
    else:
        L, rec_cap, Hkv = k_rec.shape[:3]
        B, stride = block_table.shape
        table = block_table.data_ptr()
    a = tq_evict_args(L, B, Hkv, k_rec.data_ptr(), v_rec.data_ptr(), k_rec.stride(0), v_rec.stride(0),
                      rec_cap, k_tail.data_ptr(), v_tail.data_ptr(), k_tail.stride(0), k_tail.shape[3],
                      n_chunks.data_ptr(), tail_start.data_ptr(), tail_len.data_ptr(), window, margin,
                      t_q, max_evict, table, stride)
    a._tensors = (k_rec, v_rec, k_tail, v_tail, n_chunks, tail_start, tail_len, block_table)
    return a


def tq_evict(k_codec: Codec, v_codec: Codec | None, *, stream=None, **kw):
    """Chunked eviction (arguments as make_evict_args; counters updated on the device)."""
    a = make_evict_args(**kw)
    vc = ctypes.byref(v_codec.c) if v_codec is not None else None
    _check("tq_evict", load().tq_evict(ctypes.byref(k_codec.c), vc, ctypes.byref(a), _stream(stream)))


def tq_rollback(k_codec: Codec, v_codec: Codec | None, new_len, *, stream=None, **kw):
    """Truncate every (layer, batch) stream to new_len (int32 [L, B], device) tokens; the
    cache as for tq_evict (window/margin/t_q are not used).  Counters and rings are
    updated on the device."""
    kw.setdefault("window", 0)
    kw.setdefault("margin", 0)
    a = make_evict_args(**kw)
    vc = ctypes.byref(v_codec.c) if v_codec is not None else None
    _check("tq_rollback", load().tq_rollback(ctypes.byref(k_codec.c), vc, ctypes.byref(a), _ptr(new_len),
                                             _stream(stream)))


def make_attn_args(*, q, out, scale: float, k_rec=None, v_rec=None, k_tail=None, v_tail=None,
                   n_chunks=None, tail_start=None, tail_len=None, max_chunks: int = 0,
                   max_tail: int = 0, splits: int = 0, n_kv_heads: int | None = None,
                   cuda_core_path: bool | int = False, softcap: float = 0.0, block_table=None,
                   sparse_v_eps: float = 0.0) -> tq_attn_args:
    """Build tq_attn_args from tensors.
    q: bf16 [L, B, Hq, d] (head and dim axes packed); out: f32 [L, B, Hq, d] contiguous;
    k_rec/v_rec: uint8 [L, B, Hkv, rec_cap, bytes], or with block_table (int32 [B, table_stride])
    per-layer pools uint8 [L, n_blocks, Hkv, bytes]; k_tail/v_tail: bf16 [L, B, Hkv, cap, d];
    counters int32 [L, B]; softcap > 0 caps each logit to softcap * tanh(logit / softcap)."""
    L, B, Hq, d = q.shape
    assert q.stride(3) == 1 and q.stride(2) == d, "query heads and dims must be packed"
    assert out.is_contiguous() and tuple(out.shape) == (L, B, Hq, d)
    src = k_rec if k_rec is not None else k_tail
    paged = block_table is not None
    Hkv = n_kv_heads if n_kv_heads is not None else (src.shape[2] if not (paged and k_rec is not None)
                                                     else k_rec.shape[2])
    a = tq_attn_args()
    a.n_layers, a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.scale = L, B, Hq, Hkv, d, scale
    a.q, a.q_layer_stride, a.q_batch_stride = q.data_ptr(), q.stride(0), q.stride(1)
    a.out = out.data_ptr()
    if k_rec is not None:
        a.k_rec, a.v_rec = k_rec.data_ptr(), v_rec.data_ptr()
        a.k_rec_layer_stride, a.v_rec_layer_stride = k_rec.stride(0), v_rec.stride(0)
        a.rec_cap = k_rec.shape[1] if paged else k_rec.shape[3]
    if paged:
        a.block_table, a.table_stride = block_table.data_ptr(), block_table.shape[1]
    if k_tail is not None:
        a.k_tail, a.v_tail = k_tail.data_ptr(), v_tail.data_ptr()
        a.tail_layer_stride, a.tail_cap = k_tail.stride(0), k_tail.shape[3]
    a.n_chunks = _ptr(n_chunks)
    a.tail_start = _ptr(tail_start)
    a.tail_len = _ptr(tail_len)
    a.max_chunks, a.max_tail, a.splits = max_chunks, max_tail, splits
    a.cuda_core_path = int(cuda_core_path)  # 0 automatic, 1 CUDA cores, 2 no tcgen05
    a.softcap = softcap
    a.sparse_v_eps = sparse_v_eps
    # the struct holds raw device pointers: keep the tensors alive with it
    a._tensors = (q, out, k_rec, v_rec, k_tail, v_tail, n_chunks, tail_start, tail_len, block_table)
    return a


def tq_decode_attn_plan(args: tq_attn_args, k_codec, v_codec) -> dict:
    """The kernels, split counts and launches tq_decode_attn would use (host
    only).  Codecs are Codec objects or raw tq_codec structs."""
    raw = lambda c: None if c is None else ctypes.byref(c.c if isinstance(c, Codec) else c)
    p = tq_attn_plan()
    _check("tq_decode_attn_plan", load().tq_decode_attn_plan(ctypes.byref(args), raw(k_codec), raw(v_codec),
                                                             ctypes.byref(p)))
    d = {f: getattr(p, f) for f, _ in tq_attn_plan._fields_}
    d["compressed_kernel"] = ATTN_KERNELS[d["compressed_kernel"]]
    d["dense_kernel"] = ATTN_KERNELS[d["dense_kernel"]]
    return d


def tq_decode_attn_workspace_size(args: tq_attn_args, k_codec: Codec | None, v_codec: Codec | None) -> int:
    kc = ctypes.byref(k_codec.c) if k_codec is not None else None
    vc = ctypes.byref(v_codec.c) if v_codec is not None else None
    n = load().tq_decode_attn_workspace_size(ctypes.byref(args), kc, vc)
    if n == 0:
        raise TqError("tq_decode_attn_workspace_size", TQ_ERR_INVALID_ARG)
    return int(n)


def tq_decode_attn(args: tq_attn_args, k_codec: Codec | None, v_codec: Codec | None, workspace,
                   stream=None):
    kc = ctypes.byref(k_codec.c) if k_codec is not None else None
    vc = ctypes.byref(v_codec.c) if v_codec is not None else None
    _check("tq_decode_attn", load().tq_decode_attn(ctypes.byref(args), kc, vc, _ptr(workspace),
                                                   workspace.numel() * workspace.element_size(),
                                                   _stream(stream)))


def tq_decode_attn_noalloc(args: tq_attn_args, k_codec: Codec | None, v_codec: Codec | None,
                           stream=None):
    """tq_decode_attn with the library's own fixed workspace (no allocation by
    caller or library).  Calls that overlap on the GPU share that workspace and
    race."""
    kc = ctypes.byref(k_codec.c) if k_codec is not None else None
    vc = ctypes.byref(v_codec.c) if v_codec is not None else None
    _check("tq_decode_attn_noalloc", load().tq_decode_attn_noalloc(ctypes.byref(args), kc, vc,
                                                                   _stream(stream)))


def decode_attn(*, k_codec=None, v_codec=None, workspace=None, stream=None, **kw):
    """Convenience: build the arguments, size/allocate the workspace if not given, run."""
    import torch
    a = make_attn_args(**kw)
    need = tq_decode_attn_workspace_size(a, k_codec, v_codec)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=kw["q"].device)
    tq_decode_attn(a, k_codec, v_codec, workspace, stream)
    return workspace
