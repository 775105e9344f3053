"""bench.py's GPU arm on short runs: one JSON line with the contract's keys (roofline, e2e,
kernel launch count, clocks), for a quantise + GEMM workload and for the bf16 RoPE workload
(whose step is the projection kernel alone)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(workload):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", workload, "--steps", "3",
                        "--warmup", "3", "--no-cpu-baseline"], capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,launches_per_step", [
    ("dense_mxfp8_m256_n256_k256_l1", 3),          # quantise A, quantise B, GEMM
    ("rope_proj_bf16_t16384_q1536_h128_d192", 1),  # the projection kernel alone
])
def test_bench_line(lib, workload, launches_per_step):
    d = _bench(workload)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == workload
    assert d["gpu_launches"] == launches_per_step * 3
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0


def test_per_config_records(lib):
    """The per-config GEMM records of the default run, on the small dense workload and a small
    grouped one: each frac reproduces from its GEMM time, the graph latency of config 1 is there."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    peaks, src = bench.load_peaks()
    recs = bench.per_config_records(torch.device("cuda", 0), peaks, src,
                                    entries=(("1", W.DENSE_MXFP8_256.name, True),
                                             ("5 small", W.GROUPED_FP8D_E32.name, True),
                                             ("5 small (C = NULL)", W.GROUPED_FP8D_E32.name, False)))
    assert [r["config"] for r in recs] == ["1", "5 small", "5 small (C = NULL)"]
    for r in recs:
        assert r["gemm_ms"] > 0 and r["calls"] >= 20
        assert abs(r["tflops"] - r["flops"] / (r["gemm_ms"] * 1e-3) / 1e12) <= 0.1 + 1e-3 * r["tflops"]
        assert abs(r["frac"] - r["tflops"] / r["peak"]) < 1e-3
        assert "clocks" in r
    assert recs[0]["gbs"] > 0 and recs[0]["us_per_call_graph"] > 0
    assert recs[1]["useful_tflops"] < recs[1]["tflops"] and recs[2]["c"] is None
