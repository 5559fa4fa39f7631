"""The bench's reference arm (the oracle timed on the host cores) runs without a
GPU and prints one JSON line with the keys the measurement contract asks for;
the codec workloads' byte accounting follows the record layout."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", [None, "codec_roundtrip_4096x128_b3", "encode_sweep_16M"])
def test_reference_arm_json_line(workload):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"]
    if workload:
        cmd += ["--workload", workload]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == (workload or "batched_b32_ctx32768")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_codec_workload_bytes():
    """The codec round trip moves 4096 x 256 B of bf16 in, 32 records of
    128 x 52 B (212,992 B) out, and decodes them to 2 MiB of f32; at head dim
    512 and 4 bits a vector takes 260 B (256 packed + one f32 norm); the sweep
    reads 2 to 16 GiB of bf16 per item."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    c1 = synth.CONFIGS["codec_roundtrip_4096x128_b3"]
    assert bench.codec_items(c1) == [(128, 3)]
    assert bench.codec_bytes(128, 3, 4096) == {"enc_in": 1 << 20, "enc_out": 212_992, "dec_in": 212_992,
                                               "dec_out": 2 << 20}
    assert bench.codec_bytes(512, 4, 1)["enc_out"] == 260
    sweep = synth.CONFIGS["encode_sweep_16M"]
    items = bench.codec_items(sweep)
    assert len(items) == 12 and set(items) == {(d, b) for d in (64, 128, 256, 512) for b in (2, 3, 4)}
    ins = sorted({bench.codec_bytes(d, b, sweep["n"])["enc_in"] for d, b in items})
    assert ins == [2 << 30, 4 << 30, 8 << 30, 16 << 30]
