"""bench.py's arms on the CPU: the multi-GPU refusal of the GPU arm, the
reference arm's line (rank 0 only under torchrun), and the clock record."""
import json
import os
import subprocess
import sys

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_gpu_arm_refuses_multi_gpu_runs_before_touching_cuda():
    """The library's kernels use cluster-multicast copies, so the GPU arm runs
    on one GPU only: WORLD_SIZE > 1 or --gpus > 1 exits non-zero, before
    torch (and with it CUDA) is even imported."""
    code = ("import sys; sys.argv = ['bench.py'] + sys.argv[1:]\n"
            "import bench\n"
            "try:\n"
            "    bench.main()\n"
            "except SystemExit as e:\n"
            "    print('exit', e.code, 'torch' in sys.modules)\n")
    out = _run(code, {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert out.stdout.strip().endswith("exit 2 False"), (out.stdout, out.stderr)
    assert "one GPU only" in out.stderr
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600,
                         env={k: v for k, v in os.environ.items() if k != "WORLD_SIZE"})
    assert out.returncode == 2 and "one GPU only" in out.stderr


def test_multi_gpu_request_reasons():
    class A:
        gpus = 1
    assert bench.multi_gpu_request(A, {}) is None
    assert bench.multi_gpu_request(A, {"WORLD_SIZE": "1"}) is None
    assert "WORLD_SIZE 4" in bench.multi_gpu_request(A, {"WORLD_SIZE": "4"})
    A.gpus = 8
    assert "--gpus 8" in bench.multi_gpu_request(A, {})


def test_busy_fraction():
    # two CTAs on two SMs: one busy the whole span, one half of it
    st = np.array([[0, 1, 5, 100], [0, 1, 5, 50]], dtype=np.int64)
    r = bench.sm_busy_fraction(st, 2)
    assert abs(r["sm_busy_frac"] - 0.75) < 1e-12 and r["span_us"] == 0.1


def test_clock_samples_by_phase():
    lines = [
        "2026/12/03 10:00:00.000, 0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 10:00:00.100, 0, 1900, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 10:00:00.200, 0, 1800, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 10:00:00.300, 0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    cs = bench.ClockSampler(None)
    cs.samples = cs.parse(lines)
    assert len(cs.samples) == 4
    t = [x[0] for x in cs.samples]
    all_ = cs.summary()
    assert all_["samples"] == 4 and all_["reasons"] == ["sw_power_cap"]
    assert all_["sm_mhz"] == 1900.0          # the three samples above half the peak power
    ph = cs.summary(t[1] - 0.01, t[2] + 0.01)
    assert ph["samples"] == 2 and ph["sm_mhz"] == 1850.0
    # a window between two samples takes the samples around it
    near = cs.summary(t[2] + 0.02, t[2] + 0.03)
    assert near["samples"] >= 2
    assert bench.ClockSampler(None).summary()["samples"] == 0


def test_roofline_bound_per_workload():
    pk = {"bf16_tflops": 1873.2, "hbm_gbs": 6697.5}
    sq = dict(M=8192, N=8192, K=8192)
    b, ach, peak, unit = bench.roofline_of(sq, 1.0, pk)
    assert b == "tensor" and unit == "TFLOP/s" and abs(ach - 2 * 8192 ** 3 / 1e-3 / 1e12) < 1e-6
    sk = dict(M=64, N=8192, K=8192)
    b, ach, peak, unit = bench.roofline_of(sk, 0.029, pk)
    alg = 2.0 * (64 * 8192 + 8192 * 8192 + 64 * 8192)
    assert b == "hbm" and unit == "GB/s" and peak == 6697.5
    assert abs(ach - alg / 0.029e-3 / 1e9) < 1e-6


def _bench(args, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line_on_rank_zero_only():
    """bench.py --impl reference times the CPU oracle on the host; rank 0 prints
    the contract's line, any other rank exits 0 without work."""
    args = ["--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "square512_f16",
            "--reference-rows", "8"]
    lines = _bench(args, {"RANK": "0", "WORLD_SIZE": "1"})
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "square512_f16"
    assert _bench(args, {"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_burst_clock_and_cpulist_helpers():
    # two launches x two CTAs: 1000 ns at 2000 and 1800 cycles per us
    st = np.zeros((2, 2, 6), dtype=np.int64)
    st[:, :, 3] = 1000
    st[0, :, 5] = 2000
    st[1, :, 5] = 1800
    assert bench.burst_sm_mhz(st) == [2000.0, 1800.0]
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("") == set()
