"""The C-ABI library builds, loads and exports every entry point include/tq.h
declares; host-side validation rejects bad arguments with a status (no silent
no-op, no launch).  Runs without a GPU: only calls that fail validation before
touching the device are made here."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")


@pytest.fixture(scope="module")
def lib():
    from rotated_lloyd_max_gb300 import build
    path = build.build()
    import rotated_lloyd_max_gb300 as tq
    return tq, ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b(tq_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_calls():
    names = declared_functions()
    for want in ["tq_make_codebook", "tq_encode", "tq_decode", "tq_evict", "tq_decode_attn",
                 "tq_decode_attn_workspace_size", "tq_decode_attn_plan", "tq_record_bytes",
                 "tq_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    _, raw = lib
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in tq.h but not exported"


def test_status_strings(lib):
    tq, _ = lib
    for s in range(5):
        assert tq.status_string(s).startswith("TQ_")
    assert tq.load().tq_version() >= 10000


def _codec(tq, d=128, bits=3, T=0.0, cap=0):
    c = tq.tq_codec()
    c.head_dim, c.bits, c.outlier_T, c.outlier_cap = d, bits, T, cap
    if not 1 <= bits <= 4:
        return c
    K = 1 << bits
    # a valid symmetric ascending table (values are irrelevant to validation)
    for k in range(K):
        c.centroids[k] = (k - (K - 1) / 2) / 10
    for k in range(K - 1):
        c.boundaries[k] = (c.centroids[k] + c.centroids[k + 1]) / 2
    c.boundaries[K // 2 - 1] = 0.0
    return c


def test_record_bytes_and_rejections(lib):
    tq, raw = lib
    L = tq.load()
    assert L.tq_record_bytes(ctypes.byref(_codec(tq, 128, 3))) == 128 * 52
    assert L.tq_record_bytes(ctypes.byref(_codec(tq, 512, 4))) == 128 * 260
    assert L.tq_record_bytes(ctypes.byref(_codec(tq, 128, 4, 2.0, 1312))) == 128 * 68 + 128 + 4 * 1312
    for bad in [_codec(tq, 96, 3), _codec(tq, 320, 3), _codec(tq, 128, 5), _codec(tq, 128, 0)]:
        assert L.tq_record_bytes(ctypes.byref(bad)) == 0
    asym = _codec(tq, 128, 2)
    asym.boundaries[0] = asym.boundaries[0] * 0.9
    assert L.tq_record_bytes(ctypes.byref(asym)) == 0
    bad_cap = _codec(tq, 128, 3, 2.0, 6)   # not a multiple of 4
    assert L.tq_record_bytes(ctypes.byref(bad_cap)) == 0


def test_record_bytes_match_the_oracle_layout(lib, orc):
    """The library's record size equals the oracle's (an independent
    implementation of the same layout) at every head dim and bit width, with
    and without outlier side lists (the default capacity and an odd one)."""
    import math
    tq, _ = lib
    L = tq.load()
    for d in (64, 128, 256, 512):
        for bits in (1, 2, 3, 4):
            for T, cap in ((0.0, 0), (2.0, 4 * math.ceil(0.08 * 128 * d / 4)), (1.5, 100)):
                got = L.tq_record_bytes(ctypes.byref(_codec(tq, d, bits, T, cap)))
                want = orc.Codec(d=d, bits=bits, T=T, cap=cap).record_bytes
                assert got == want, (d, bits, T, cap, got, want)
                assert got % 16 == 0


def test_calls_fail_loudly_on_bad_arguments(lib):
    tq, _ = lib
    L = tq.load()
    good = _codec(tq, 128, 3)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    # unsupported head dims: a status, not a silent return
    assert L.tq_encode(ctypes.byref(_codec(tq, 96, 3)), fake, 1, 128, 96, 0, fake, 0, 0, None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_decode(ctypes.byref(_codec(tq, 320, 3)), fake, 1, 128, 0, 0, fake, 320, 0, None) == tq.TQ_ERR_UNSUPPORTED
    # null / misaligned pointers, bad strides
    assert L.tq_encode(ctypes.byref(good), None, 1, 128, 128, 0, fake, 0, 0, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_encode(ctypes.byref(good), ctypes.c_void_p(0x10002), 1, 128, 128, 0, fake, 0, 0, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_encode(ctypes.byref(good), fake, 1, 128, 100, 0, fake, 0, 0, None) == tq.TQ_ERR_INVALID_ARG
    # outliers need record-aligned starts
    outl = _codec(tq, 128, 3, 2.0, 1312)
    assert L.tq_encode(ctypes.byref(outl), fake, 1, 10, 128, 0, fake, 0, 5, None) == tq.TQ_ERR_INVALID_ARG
    # empty work is a successful no-op that launches nothing
    assert L.tq_encode(ctypes.byref(good), fake, 0, 128, 128, 0, fake, 0, 0, None) == tq.TQ_OK
    # codebook: unsupported shapes and a too-small scratch
    out = tq.tq_codec()
    assert L.tq_make_codebook(5, 128, 1, 0.0, 0, fake, 4096, ctypes.byref(out), None, None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_make_codebook(3, 96, 1, 0.0, 0, fake, 4096, ctypes.byref(out), None, None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_make_codebook(3, 128, 1, 0.0, 0, fake, 8, ctypes.byref(out), None, None) == tq.TQ_ERR_WORKSPACE
    # attention: Hq % Hkv != 0, bad head dim, missing pointers
    a = tq.tq_attn_args()
    a.n_layers, a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.scale = 1, 1, 6, 4, 128, 1.0
    a.q, a.out = 0x10000, 0x20000
    assert L.tq_decode_attn(ctypes.byref(a), None, None, fake, 1 << 20, None) == tq.TQ_ERR_INVALID_ARG
    a.n_kv_heads, a.head_dim = 2, 96
    assert L.tq_decode_attn(ctypes.byref(a), None, None, fake, 1 << 20, None) == tq.TQ_ERR_UNSUPPORTED
    a.head_dim = 128
    a.k_rec = 0x30000   # records without codecs
    assert L.tq_decode_attn(ctypes.byref(a), None, None, fake, 1 << 20, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_decode_attn_workspace_size(ctypes.byref(a), None, None) == 0
    # soft cap: 0 (off) and positive caps are accepted, negative or non-finite ones rejected
    a.k_rec = None
    a.k_tail, a.v_tail, a.tail_cap, a.max_tail, a.tail_layer_stride = 0x30000, 0x40000, 16, 16, 2 * 16 * 128
    a.tail_start, a.tail_len = 0x50000, 0x60000
    for cap, ok in [(0.0, True), (30.0, True), (1.0, True), (-1.0, False), (float("nan"), False),
                    (float("inf"), False)]:
        a.softcap = cap
        assert (L.tq_decode_attn_workspace_size(ctypes.byref(a), None, None) > 0) == ok, cap
        if not ok:
            assert L.tq_decode_attn(ctypes.byref(a), None, None, fake, 1 << 20, None) == tq.TQ_ERR_INVALID_ARG
    # eviction: null counters
    e = tq.tq_evict_args()
    e.n_layers, e.batch, e.n_kv_heads, e.max_evict, e.rec_cap, e.tail_cap, e.t_q = 1, 1, 1, 1, 4, 272, 1
    assert L.tq_evict(ctypes.byref(good), ctypes.byref(good), ctypes.byref(e), None) == tq.TQ_ERR_INVALID_ARG


def test_evict_rejects_a_tail_that_cannot_reach_the_bound(lib):
    """The tail ring must hold window + max(t_q - 1, margin) + 128 tokens (272
    at window 128, margin 16, t_q 1); smaller rings are rejected on the host."""
    tq, L = lib
    good = tq.tq_codec()
    good.head_dim, good.bits = 128, 1
    good.centroids[0], good.centroids[1], good.boundaries[0] = -0.07, 0.07, 0.0
    e = tq.tq_evict_args()
    e.n_layers, e.batch, e.n_kv_heads, e.max_evict, e.rec_cap, e.t_q = 1, 1, 1, 1, 4, 1
    e.k_rec = e.v_rec = 0x10000
    e.k_tail = e.v_tail = 0x20000
    e.n_chunks, e.tail_start, e.tail_len = 0x30000, 0x40000, 0x50000
    e.window, e.margin, e.tail_cap = 128, 16, 271
    assert L.tq_evict(ctypes.byref(good), ctypes.byref(good), ctypes.byref(e), None) == tq.TQ_ERR_INVALID_ARG
    e.window, e.margin, e.t_q, e.tail_cap = 0x7FFFFFFF, 0, 1, 0x7FFFFFFF    # floor + 128 overflows int32
    assert L.tq_evict(ctypes.byref(good), ctypes.byref(good), ctypes.byref(e), None) == tq.TQ_ERR_INVALID_ARG


def test_noalloc_rejections_need_no_device(lib):
    """The allocation-free entry point returns the planner's status (invalid
    vs unsupported) and rejects a workspace above its fixed array before it
    touches a device."""
    tq, L = lib
    a = tq.tq_attn_args()
    a.n_layers, a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.scale = 1, 1, 6, 4, 128, 1.0
    a.q, a.out = 0x10000, 0x20000
    a.k_tail, a.v_tail, a.tail_cap, a.max_tail, a.tail_layer_stride = 0x30000, 0x40000, 8, 8, 8 * 128
    a.tail_start, a.tail_len = 0x50000, 0x60000
    assert L.tq_decode_attn_noalloc(ctypes.byref(a), None, None, None) == tq.TQ_ERR_INVALID_ARG   # 6 % 4
    a.n_kv_heads, a.head_dim = 2, 96
    assert L.tq_decode_attn_noalloc(ctypes.byref(a), None, None, None) == tq.TQ_ERR_UNSUPPORTED
    a.head_dim = 512
    a.n_layers, a.batch, a.n_q_heads, a.n_kv_heads = 64, 64, 64, 1   # 64^3 rows x 512 floats > 8 MiB
    a.tail_layer_stride = 64 * 8 * 512
    assert L.tq_decode_attn_workspace_size(ctypes.byref(a), None, None) > tq.NOALLOC_WORKSPACE_BYTES
    assert L.tq_decode_attn_noalloc(ctypes.byref(a), None, None, None) == tq.TQ_ERR_WORKSPACE


def test_struct_layouts_match_header(lib, tmp_path):
    """The ctypes mirrors of the C structs have the C compiler's size and field
    offsets (checked by compiling a probe against include/tq.h with gcc)."""
    import subprocess
    tq, _ = lib
    structs = {"tq_codec": tq.tq_codec, "tq_evict_args": tq.tq_evict_args, "tq_attn_args": tq.tq_attn_args,
               "tq_attn_plan": tq.tq_attn_plan}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} %zu\\n", sizeof({name}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{name}.{fname} %zu\\n", offsetof({name}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", str(src), "-o", str(exe)])
    got = dict(l.split() for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert int(got[f"{name}.{fname}"]) == getattr(cls, fname).offset, f"{name}.{fname}"


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "tq.h"

/* A plain C caller of the boundary: host-only calls, fake aligned device
 * addresses that are never dereferenced.  The 6 bf16 layers of the
 * Qwen2-shaped cache as one dense call. */
int main(void) {
  tq_attn_args a;
  tq_attn_plan p;
  memset(&a, 0, sizeof(a));
  a.n_layers = 6; a.batch = 1; a.n_q_heads = 12; a.n_kv_heads = 2; a.head_dim = 128; a.scale = 1.0f;
  a.q = (const void*)0x100000; a.out = (float*)0x200000;
  a.q_layer_stride = 12 * 128; a.q_batch_stride = 12 * 128;
  a.k_tail = (const void*)0x300000; a.v_tail = (const void*)0x400000;
  a.tail_layer_stride = 2 * 2048 * 128; a.tail_cap = 2048; a.max_tail = 2048;
  a.tail_start = (const int32_t*)0x500000; a.tail_len = (const int32_t*)0x600000;
  if (tq_version() < 10000) return 2;
  tq_status st = tq_decode_attn_plan(&a, NULL, NULL, &p);
  if (st != TQ_OK) { printf("%s\n", tq_status_string(st)); return 3; }
  if ((size_t)p.workspace_bytes != tq_decode_attn_workspace_size(&a, NULL, NULL)) return 4;
  printf("%d %d %d %d %d\n", p.compressed_kernel, p.dense_kernel, p.dense_splits, p.dense_tokens_per_split,
         p.launches);
  a.head_dim = 96;
  return tq_decode_attn_plan(&a, NULL, NULL, &p) == TQ_ERR_UNSUPPORTED ? 0 : 5;
}
"""


def test_plain_c_client_links_and_plans(lib, tmp_path):
    """The library serves a C program (gcc, no Python): it links against
    libtq_gb300.so with include/tq.h and gets the planner's answer: 6 layers x 2 kv
    heads want ceil(16 x 152 / 12) = 203 splits, capped at the 64 tiles of 32
    tokens and then at 256 tokens per split: 8 dense splits on mma.sync."""
    import subprocess
    from rotated_lloyd_max_gb300 import build
    so = build.build()
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(so)
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(so), "-Wl,-rpath," + libdir])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.split() == ["0", "3", "8", "256", "2"]


def test_no_cpu_fallback_without_the_library(tmp_path):
    """Without libtq_gb300.so every entry point raises (no silent CPU path):
    a fresh interpreter whose package points at a missing library."""
    import subprocess
    import sys
    code = (
        "import rotated_lloyd_max_gb300 as tq\n"
        "tq.LIB_PATH = %r\n"
        "for call in (lambda: tq.load(), lambda: tq.tq_record_bytes(tq.Codec(c=tq.tq_codec(), mse=0.0))):\n"
        "    try:\n"
        "        call()\n"
        "    except ImportError as e:\n"
        "        assert 'no CPU fallback' in str(e)\n"
        "    else:\n"
        "        raise SystemExit('no error')\n"
        "print('ok')\n" % str(tmp_path / "absent" / "libtq_gb300.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.stdout, r.stderr[-2000:])


def _gauss_codec(tq, orc, bits, d):
    c = tq.tq_codec()
    c.head_dim, c.bits, c.sign_seed = d, bits, 1
    cent, bnd = orc.codebook_f32(bits, d)
    for k, v in enumerate(cent):
        c.centroids[k] = float(v)
    for k, v in enumerate(bnd):
        c.boundaries[k] = float(v)
    return tq.Codec(c, 0.0)


def test_set_centroids_fills_midpoints_and_validates(lib, orc):
    """tq_codec_set_centroids (host only): a caller's symmetric ascending table
    replaces the Gaussian one with the same f32 midpoints the oracle derives;
    unordered, non-finite, asymmetric, too-large and too-close tables are
    rejected and leave the codec unchanged."""
    import numpy as np
    tq, _ = lib
    d, bits = 128, 3
    base = _gauss_codec(tq, orc, bits, d)
    half = np.float32(np.array([0.1, 0.35, 0.7, 1.3]) / math.sqrt(d))
    tab = [float(v) for v in np.concatenate([-half[::-1], half])]
    c = tq.tq_codec_set_centroids(base, tab)
    assert c.centroids() == [float(np.float32(v)) for v in tab]
    np.testing.assert_array_equal(np.array(c.boundaries(), np.float32), orc.midpoints_f32(bits, np.array(tab, np.float32)))
    assert tq.tq_record_bytes(c) == base.record_bytes
    bad = {
        "unordered": tab[:3] + [tab[4], tab[3]] + tab[5:],
        "nan": tab[:7] + [float("nan")],
        "asymmetric": tab[:7] + [tab[7] * 1.01],
        "too large": [v * 12.0 for v in tab],
        "too close": [v * 0.02 for v in tab],
        "wrong count": tab[:4],
    }
    want = {"unordered": tq.TQ_ERR_INVALID_ARG, "nan": tq.TQ_ERR_INVALID_ARG, "wrong count": tq.TQ_ERR_INVALID_ARG,
            "asymmetric": tq.TQ_ERR_UNSUPPORTED, "too large": tq.TQ_ERR_UNSUPPORTED,
            "too close": tq.TQ_ERR_UNSUPPORTED}
    for name, t in bad.items():
        with pytest.raises(tq.TqError) as e:
            tq.tq_codec_set_centroids(base, t)
        assert e.value.status == want[name], name
    # two-bit tables have no cell-spacing condition
    c2 = tq.tq_codec_set_centroids(_gauss_codec(tq, orc, 2, d), [-0.02, -0.001, 0.001, 0.02])
    assert c2.boundaries()[1] == 0.0


def test_scale_mode_is_validated(lib, orc):
    tq, _ = lib
    c = _gauss_codec(tq, orc, 3, 128)
    for m in range(4):
        c.c.scale_mode = m
        assert tq.load().tq_record_bytes(ctypes.byref(c.c)) > 0
    c.c.scale_mode = 4
    assert tq.load().tq_record_bytes(ctypes.byref(c.c)) == 0
