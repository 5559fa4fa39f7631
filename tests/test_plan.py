"""The attention planner (host code, no GPU): tq_decode_attn_plan reports the
kernels, split counts and launches tq_decode_attn uses; the values here follow
from the planning rules by hand, at GB300's 152 SMs (the count the planner
takes when no device is visible)."""
import ctypes
import math

import pytest

import rotated_lloyd_max_gb300 as tq

ALIGNED = 0x100000   # fake, 256-byte aligned device addresses: nothing is dereferenced


def _addr(i):
    return ALIGNED * (i + 1)


def raw_codec(orc, bits, d, T=0.0):
    """A tq_codec holding the oracle's f32 table (the device codebook kernel
    needs a GPU)."""
    c = tq.tq_codec()
    c.head_dim, c.bits, c.sign_seed, c.outlier_T = d, bits, 1, T
    c.outlier_cap = 4 * math.ceil(0.08 * 128 * d / 4) if T else 0
    cent, bnd = orc.codebook_f32(bits, d)
    for k, v in enumerate(cent):
        c.centroids[k] = float(v)
    for k, v in enumerate(bnd):
        c.boundaries[k] = float(v)
    return c


def args_for(*, L, B, Hq, Hkv, d, records=0, tail=0, shared=False, splits=0, path=0, rec_bytes=0):
    a = tq.tq_attn_args()
    a.n_layers, a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.scale = L, B, Hq, Hkv, d, 1.0
    a.q, a.out = _addr(0), _addr(1)
    a.q_layer_stride, a.q_batch_stride = B * Hq * d, Hq * d
    if records:
        a.k_rec = _addr(2)
        a.v_rec = a.k_rec if shared else _addr(3)
        a.k_rec_layer_stride = a.v_rec_layer_stride = B * Hkv * records * rec_bytes
        a.rec_cap, a.max_chunks, a.n_chunks = records, records, _addr(4)
    if tail is not None:
        cap = max(tail, 1)
        a.k_tail = _addr(5)
        a.v_tail = a.k_tail if shared else _addr(6)
        a.tail_layer_stride, a.tail_cap, a.max_tail = B * Hkv * cap * d, cap, tail
        a.tail_start, a.tail_len = _addr(7), _addr(8)
    a.splits, a.cuda_core_path = splits, path
    return a


def plan(a, kc, vc):
    p = tq.tq_decode_attn_plan(a, kc, vc)
    assert p["workspace_bytes"] == tq.load().tq_decode_attn_workspace_size(
        ctypes.byref(a), ctypes.byref(kc) if kc else None, ctypes.byref(vc) if vc else None)
    return p


@pytest.fixture(scope="module")
def c4_512(orc):
    return raw_codec(orc, 4, 512)


def test_v4flash_mqa_plan(orc, c4_512):
    """43 layers x 510 records + 256 tail tokens, 64 heads on one kv head: the
    tcgen05 kernel at 7 splits of 73 records (the one-CTA-per-SM cost model:
    2 waves x 75 = 150 against 156-174 for its neighbours), the tail in 2 splits
    of 128 tokens on the mma.sync dense kernel (16 heads per CTA), then the merge."""
    a = args_for(L=43, B=1, Hq=64, Hkv=1, d=512, records=510, tail=256, shared=True, rec_bytes=128 * 260)
    p = plan(a, c4_512, c4_512)
    assert p["compressed_kernel"] == "tcgen05" and p["dense_kernel"] == "mma512"
    assert (p["compressed_splits"], p["records_per_split"]) == (7, 73)
    assert (p["dense_splits"], p["dense_tokens_per_split"]) == (2, 128)
    assert (p["heads_per_cta"], p["dense_heads_per_cta"], p["launches"]) == (64, 16, 3)


def test_d512_dense_splits_fall_back_for_groups_off_sixteen(orc, c4_512):
    """24 heads a kv head: tcgen05 for the records, but the tail's CTAs need
    groups of 16 heads on the tensor cores, so it runs 8-head CUDA-core CTAs."""
    a = args_for(L=2, B=1, Hq=24, Hkv=1, d=512, records=20, tail=256, shared=True, rec_bytes=128 * 260)
    p = plan(a, c4_512, c4_512)
    assert (p["compressed_kernel"], p["dense_kernel"], p["dense_heads_per_cta"]) == ("tcgen05", "cuda_core", 8)


def test_v4flash_mqa_other_paths(orc, c4_512):
    a = args_for(L=43, B=1, Hq=64, Hkv=1, d=512, records=510, tail=256, shared=True, rec_bytes=128 * 260,
                 path=2)
    p = plan(a, c4_512, c4_512)          # no tcgen05: mma.sync with 16-head CTAs
    assert p["compressed_kernel"] == "mma512" and p["heads_per_cta"] == 16 and p["launches"] == 3
    a.cuda_core_path = 1                  # CUDA cores only: one launch of 8-head CTAs + the merge
    p = plan(a, c4_512, c4_512)
    assert (p["compressed_kernel"], p["dense_kernel"], p["heads_per_cta"], p["launches"]) == \
        ("cuda_core", "cuda_core", 8, 2)


def test_explicit_splits_are_kept(orc, c4_512):
    """splits = 5: 5 splits of 102 records; the tail's 32 tiles of 8 tokens in
    splits of 7 tiles (56 tokens), 5 of them."""
    a = args_for(L=43, B=1, Hq=64, Hkv=1, d=512, records=510, tail=256, shared=True, rec_bytes=128 * 260,
                 splits=5)
    p = plan(a, c4_512, c4_512)
    assert (p["compressed_splits"], p["records_per_split"]) == (5, 102)
    assert (p["dense_splits"], p["dense_tokens_per_split"]) == (5, 56)


def test_qwen2_plan(orc):
    """28 layers (22 with 16 records, 6 bf16 with 2048 dense tokens) in one call:
    56 units want ceil(16 x 152 / 56) = 44 splits; the tensor-core kernel takes
    at least 2 records and 256 dense tokens per split: 8 x 2 records and
    8 x 256 tokens, one launch of 6-head CTAs + the merge."""
    kc, vc = raw_codec(orc, 3, 128), raw_codec(orc, 2, 128)
    a = args_for(L=28, B=1, Hq=12, Hkv=2, d=128, records=16, tail=2048, rec_bytes=128 * 52)
    p = plan(a, kc, vc)
    assert p["compressed_kernel"] == p["dense_kernel"] == "mma"
    assert (p["compressed_splits"], p["records_per_split"]) == (8, 2)
    assert (p["dense_splits"], p["dense_tokens_per_split"]) == (8, 256)
    assert (p["heads_per_cta"], p["launches"]) == (6, 2)


def test_outlier_codecs_take_the_warp_local_kernel_and_sparse_v_the_tensor_cores(orc):
    """Side lists run on the warp-local CUDA-core kernel; with sparse-V on the
    tensor-core kernel in CTAs of three 4-warp groups (one CTA per SM, one
    copy of the 4-bit pair table: the batched cache's codecs need 220 KB of
    shared memory for that).  Dense splits of such a call run in a second
    launch of 4-warp CTAs."""
    kc, vc = raw_codec(orc, 4, 128, T=2.0), raw_codec(orc, 3, 128, T=2.0)
    a = args_for(L=1, B=32, Hq=32, Hkv=8, d=128, records=256, tail=None, rec_bytes=8192)
    p = plan(a, kc, vc)
    assert p["compressed_kernel"] == "cuda_core_warp" and p["dense_kernel"] == "none"
    assert (p["heads_per_cta"], p["warps_per_cta"], p["launches"]) == (4, 4, 2)
    a.sparse_v_eps = 1e-3
    p = plan(a, kc, vc)
    assert p["compressed_kernel"] == "mma" and p["dense_kernel"] == "none"
    assert (p["heads_per_cta"], p["warps_per_cta"], p["launches"]) == (4, 12, 2)
    b = args_for(L=1, B=2, Hq=8, Hkv=2, d=128, records=4, tail=64, rec_bytes=8192)
    b.sparse_v_eps = 1e-3
    p = plan(b, kc, vc)
    assert p["compressed_kernel"] == p["dense_kernel"] == "mma"
    assert (p["warps_per_cta"], p["launches"]) == (12, 3)


def test_codecs_without_side_lists_keep_four_warp_ctas(orc):
    kc, vc = raw_codec(orc, 4, 128), raw_codec(orc, 3, 128)
    a = args_for(L=1, B=32, Hq=32, Hkv=8, d=128, records=256, tail=None, rec_bytes=8192)
    p = plan(a, kc, vc)
    assert p["compressed_kernel"] == "mma" and p["warps_per_cta"] == 4 and p["launches"] == 2


def test_head_dim_256_runs_on_cuda_cores(orc):
    c = raw_codec(orc, 2, 256)
    a = args_for(L=1, B=1, Hq=4, Hkv=4, d=256, records=3, tail=70, rec_bytes=128 * 68)
    p = plan(a, c, c)
    assert p["compressed_kernel"] == p["dense_kernel"] == "cuda_core"


def test_codec_objects_are_accepted(orc, c4_512):
    """The binding takes Codec objects (as tq_make_codebook returns them) as
    well as raw tq_codec structs, with the same plan."""
    a = args_for(L=43, B=1, Hq=64, Hkv=1, d=512, records=510, tail=256, shared=True, rec_bytes=128 * 260)
    wrapped = tq.Codec(c=c4_512, mse=0.0)
    assert tq.tq_decode_attn_plan(a, wrapped, wrapped) == tq.tq_decode_attn_plan(a, c4_512, c4_512)


def test_empty_context_is_one_dense_split():
    a = args_for(L=1, B=2, Hq=4, Hkv=2, d=128, tail=0)
    p = plan(a, None, None)
    assert p["compressed_kernel"] == "none" and p["dense_kernel"] == "mma"
    assert (p["compressed_splits"], p["dense_splits"], p["launches"]) == (0, 1, 2)


def test_plan_rejects_what_the_call_rejects(orc):
    a = args_for(L=1, B=1, Hq=6, Hkv=4, d=128, tail=16)
    with pytest.raises(tq.TqError):
        tq.tq_decode_attn_plan(a, None, None)
    a = args_for(L=1, B=1, Hq=8, Hkv=4, d=128, tail=16)
    assert tq.load().tq_decode_attn_plan(ctypes.byref(a), None, None, None) == 1   # TQ_ERR_INVALID_ARG
