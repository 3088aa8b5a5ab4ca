"""The benchmark's JSON line on the GPU: one line with every key of the
contract, run on a reduced key length so that it finishes in seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--kv-len", "16384",
                        "--steps", "3", "--warmup", "3", "--no-cpu-baseline"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["roofline"]["bound"] == "tensor" and d["roofline"]["achieved"] > 0
    assert d["roofline"]["peak"] > 0
    # the kernel is timed in steps of tens of milliseconds: the burst peak
    roof = d["roofline"]
    assert roof["peak_kind"].startswith("bf16_tflops burst")
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert "clocks" in d["e2e"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * 3
    assert "sm_mhz" in d["clocks"]


def test_all_configs_prints_gpu_beside_oracle_for_every_workload():
    """bench.py --all-configs: one line per workload with the GPU time and,
    from the same run, the oracle's time on the host cores."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--all-configs"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.strip()]
    assert [d["workload"] for d in lines] == ["c1", "c2", "c3", "c4", "c5"]
    for d in lines:
        assert d["gpu_ms"] > 0 and d["gpu_tflops"] > 0
        o = d["oracle"]
        assert o["seconds"] > 0 and o["cores"] >= 1 and o["kind"] == "oracle" and o["sample"]


def test_measure_reports_graph_replay_times():
    """measure.py --graph: each line carries the per-call time of the same
    calls replayed from one CUDA graph; for the 1,024-token launch the host
    submits slower than the device runs, so the replay is the faster one."""
    r = subprocess.run([sys.executable, "-m", "ring_attention_attn_gb300.measure", "--path",
                        "ring_c1", "merge", "--reps", "10", "--graph"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.strip()]
    assert [l["path"] for l in lines] == ["ring_c1", "merge"]
    for l in lines:
        assert l["ms"] > 0 and l["graph_ms"] is not None and l["graph_ms"] > 0
        assert abs(l["graph_achieved"] - l["achieved"] * l["ms"] / l["graph_ms"]) < 1e-6 * l[
            "graph_achieved"]
    assert lines[0]["graph_ms"] < lines[0]["ms"]
