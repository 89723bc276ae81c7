"""bench.py's own arm on a small case (2 of the 36 layers): one JSON line with
the contract's keys - roofline of the dominant kernel against the measured
peak, the end-to-end leg through host buffers with its byte counts, the
launch count and the clock samples."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--layers", "2",
                        "--steps", "3", "--warmup", "3", "--legs", "device,e2e", "--e2e-steps", "2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "gpu_launches", "clocks", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"].startswith("qwen3_8b") and d["config"]["layers"] == 2
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None          # profiles/ hold the 36-layer launch, not this one
    assert d["gpu_launches"] == 3 * 3
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "GB/s"
    src = 2 * 2 * 2048 * 16 * 8 * 128 * 2             # K and V, 2 layers, fp16
    assert e["h2d_bytes_per_step"] >= src and e["d2h_bytes_per_step"] >= src
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_per_layer_workload_objects():
    """The per-layer objects of the default line (measure_layered) on 2-layer
    cuts of the Llama-3-70B-shaped and ragged workloads: per-call medians for
    every block size, the layered pass, and the fetch target arithmetic."""
    import torch
    import bench
    import workloads
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    w = workloads.llama3_70b()
    w.L = 2
    r = bench.measure_layered(w, "fp8", dev, steps=3, warmup=3, distinct_layers=True)
    assert set(r["fetch"]) == {"B64"} and set(r["encode"]) == {"B64"}
    f = r["fetch"]["B64"]
    assert f["calls"] == 3 * 2 and f["median_us"] > 0 and f["gbs"] > 0
    assert f["bytes_per_call"] == bench.layered_bytes(w, w.blocks[0], "fp8")[1]
    assert abs(bench.fetch_target_us(402_726_912) - 71.9) < 0.05
    assert r["pass"]["gbs"] > 0 and r["pass"]["per_layer_us"] > 0
    w = workloads.ragged()
    w.L = 2
    r = bench.measure_layered(w, "int4", dev, steps=3, warmup=3)
    assert set(r["fetch"]) == {"B16", "B64"} and r["tokens"] == sum(b.tokens() for b in w.blocks)


def test_crc_leg_object():
    """`--crc` adds the CRC-32 of the step's wire and the fused slab CRC; its
    integer-ALU roofline is given only for the full launch whose ALU count
    profiles/ records, so on a 2-layer cut it is null."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--layers", "2",
                        "--steps", "3", "--warmup", "3", "--legs", "device", "--crc"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.strip().startswith("{")][-1])
    c = d["crc32"]
    assert c["kernel"] == "k_crc32" and c["units"] == 2 * 2048 and c["gbs"] > 0
    assert c["bytes_per_launch"] == 2 * 2048 * (32768 + 64)
    assert c["roofline"] is None
    f = c["fused_encode"]
    assert f["encode_with_crc_ms"] > 0 and f["encode_ms"] > 0
