"""The benchmark's JSON contract on the CPU-only reference arm (the oracle timed on the host
cores): one line with the contract's keys, the reference markers, and e2e mirroring the
line's own value; plus the host-side helpers the GPU arm's roofline uses."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                        "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_profile_traffic_matches_the_committed_source():
    sys.path.insert(0, ROOT)
    import bench

    # the committed summary carries the current streaming-kernel source hash, so the bench
    # reports its DRAM traffic; a stale hash would make it report null
    t = bench.profile_traffic("q_gemv_q4_0_decode_shapes.md")
    assert t is not None and t > 0
