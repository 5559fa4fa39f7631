"""The per-layer calls of the end-to-end pipeline (one tq_encode, tq_evict and
tq_decode_attn per layer, as a model's layer loop issues them) give the same
attention output as the whole-cache calls the bench times: the same records
and counters, and outputs within f32 summation-order noise (the two plans
split the records differently)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bench_mod():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rotated_lloyd_max_gb300 import build
    build.build()
    import bench
    return bench


@pytest.mark.parametrize("name,layers,batch", [("batched_b32_ctx32768", 2, 2), ("longctx_b4_ctx262144", 2, 1),
                                                ("v4flash_mqa_ctx65536", 3, None)])
def test_per_layer_calls_match_the_whole_cache_call(bench_mod, name, layers, batch):
    import torch
    wl = bench_mod.CacheWorkload(name, "cuda", layers=layers, batch=batch)
    wl.krec.fill_(0)            # both flows start from zeroed records (a side list's unused slots stay 0)
    wl.vrec.fill_(0)
    wl.encode()
    wl.ev.reset()
    wl.ev.run()
    wl.attention()
    torch.cuda.synchronize()
    want = wl.out.cpu().numpy().copy()
    rec_k = wl.krec.cpu().numpy().copy()
    counters = [t.cpu().numpy().copy() for t in (wl.ev.n_chunks, wl.ev.tail_start, wl.ev.tail_len)]
    rec_v = wl.vrec.cpu().numpy().copy()
    wl.out.fill_(float("nan"))
    wl.krec.fill_(0)
    wl.vrec.fill_(0)
    wl.ev.reset()
    for l in wl.comp:
        wl.encode_layer(l)
        wl.ev.run_layer(l - wl.c0)
        wl.attention_layer(l)
    torch.cuda.synchronize()
    got = wl.out.cpu().numpy()
    assert np.array_equal(wl.krec.cpu().numpy(), rec_k)
    assert np.array_equal(wl.vrec.cpu().numpy(), rec_v)
    for t, c in zip((wl.ev.n_chunks, wl.ev.tail_start, wl.ev.tail_len), counters):
        assert np.array_equal(t.cpu().numpy(), c)
    comp = np.array(wl.comp)
    assert np.all(np.isfinite(got[comp]))
    err = np.max(np.abs(got[comp] - want[comp]))
    assert err <= 1e-5 * max(1.0, float(np.max(np.abs(want[comp])))), f"max abs difference {err}"
