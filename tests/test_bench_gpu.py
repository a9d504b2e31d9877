"""bench.py end to end on the GPU, on the small workload: the JSON line carries
the contract's keys, with values that agree with one another."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_the_small_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "square512_f16",
                          "--only-headline", "--steps", "5", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "per_workload"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["gpu_launches"] == 5
    assert d["value"] > 0 and abs(d["value"] - 2 * 512 ** 3 / (d["ms_per_step"] * 1e-3) / 1e12) < 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] in ("tensor", "hbm") and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 2 * 2 * 512 * 512
    assert e["d2h_bytes_per_step"] == 2 * 512 * 512
    assert e["host_link"]["h2d_gbs"] > 0
    assert list(d["per_workload"]) == ["square512_f16"]
    w = d["per_workload"]["square512_f16"]
    assert w["best_schedule"] in w["per_schedule"] and w["priming_launches"] >= 3
    assert set(w["per_schedule"]) == {"dp", "persistent", "streamk", "streamk_all", "splitk",
                                      "splitk_cluster", "auto"}
