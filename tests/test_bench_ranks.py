"""The benchmark's multi-rank host logic (max over ranks, whole-job value) on
two gloo ranks on the CPU; no GPU is involved."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [120.0, 150.0][rank]                   # rank 1 is the slow one
    t = bench.max_over_ranks(my_ms, dist, world, "cpu")
    v = bench.whole_job_tflops(1e12, 10, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, t, v in got:
        assert t == 150.0
        assert abs(v - 2 * 10 * 1e12 / 0.150 / 1e12) < 1e-9


def test_single_rank_and_busy_fraction():
    assert bench.max_over_ranks(3.5, None, 1, "cpu") == 3.5
    # two CTAs on two SMs: one busy the whole span, one half of it
    st = np.array([[0, 1, 5, 100], [0, 1, 5, 50]], dtype=np.int64)
    r = bench.sm_busy_fraction(st, 2)
    assert abs(r["sm_busy_frac"] - 0.75) < 1e-12 and r["span_us"] == 0.1


def _bench(args, env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.update(env_extra)
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
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
