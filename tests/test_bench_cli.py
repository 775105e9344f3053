"""bench.py's reference arm (the float64 oracle on the host cores) runs without a GPU: its JSON
line carries the keys the benchmark contract names, and ranks other than 0 exit quietly."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def _line(out):
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _line(_run(["--impl", "reference", "--workload", "dense_mxfp8_m256_n256_k256_l1", "--steps", "2",
                    "--warmup", "1", "--ref-rows", "256"]))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["value"] > 0
    assert d["config"]["workload"] == "dense_mxfp8_m256_n256_k256_l1"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_bf16_rope_workload():
    d = _line(_run(["--impl", "reference", "--workload", "rope_proj_bf16_t16384_q1536_h128_d192", "--steps", "1",
                    "--warmup", "0", "--ref-rows", "256"]))
    assert d["config"]["format"] == "bf16" and d["value"] > 0
    assert "bf16 values" in d["cpu_baseline"]["sample"]


def test_reference_arm_other_ranks_print_nothing():
    out = _run(["--impl", "reference", "--workload", "dense_mxfp8_m256_n256_k256_l1", "--steps", "1",
                "--warmup", "0", "--ref-rows", "256"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_every_workload_has_a_config_and_a_bounded_oracle_sample():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    for name, wl in W.ALL.items():
        cfg = bench._config(wl)
        assert cfg["workload"] == name and cfg["flops_per_step"] == wl.flops
        assert cfg["l2"] and cfg["step"]
        rows = bench.oracle_rows(wl)
        limit = wl.tokens if isinstance(wl, W.RopeProj) else (wl.m if isinstance(wl, W.Dense) else wl.valid_m)
        assert 256 <= rows <= max(256, limit)
        assert rows % 256 == 0 or rows == limit  # whole 256-row groups, or the whole operand
        assert bench.oracle_rows(wl, 512) == 512
