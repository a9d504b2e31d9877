#!/usr/bin/env python3
"""Benchmark: GEMM TFLOP/s (device-timed) and fraction of the GB300 roofline,
per schedule, on one synthetic workload (default: bf16 8192 x 8192 x 8192,
row-major A, column-major B).

One step = one C = A*B through the C ABI (gemm_run) with the schedule that
measured fastest in an untimed-for-the-headline per-schedule pass.  Prints
one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--schedule dp|persistent|streamk|best] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 product) on the host
cores instead, on a bounded row sample of the same workload per step.
Under torchrun (N > 1) every rank runs its own copy of the workload (weak
scaling, no collective on the data path); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from persistent_stream_matmul_gb300 import inputs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6
SCHED_NAMES = ["dp", "persistent", "streamk", "streamk_all", "splitk", "auto"]
# name -> (schedule, options): "streamk" is the hybrid rule of the issue's final
# version; "streamk_all" puts every tile in the Stream-K wave
SCHED_DEFS = {"dp": ("dp", {}), "persistent": ("persistent", {}),
              "streamk": ("streamk", {}), "streamk_all": ("streamk", {"sk_mode": 1}),
              "splitk": ("splitk", {}), "auto": ("auto", {})}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "persistent_stream_matmul_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def resolved_name(name: str, plan) -> str:
    """The per-schedule name of what a plan runs: AUTO resolves to one of the
    others, and its DRAM traffic is that schedule's."""
    if name != "auto":
        return name
    kind = {0: "dp", 1: "persistent", 2: "streamk", 3: "splitk"}.get(plan.info("schedule"), "auto")
    return "streamk_all" if kind == "streamk" and plan.info("sk_mode") == 1 else kind


def profiled_traffic(workload: str, schedule: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    sources have not changed since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_kernel_%s_%s.md" % (schedule, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_id: str | None):
        self.proc = None
        self.device_id = device_id
        fd, self.path = tempfile.mkstemp(prefix="psm_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.device_id:
                cmd += ["-i", self.device_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        busy = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] if power else sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def device_pci_id(torch, dev: int):
    try:
        pr = torch.cuda.get_device_properties(dev)
        return "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        return None


# --------------------------------------------------------------------- oracle (CPU)
def oracle_rows_gflops(A, Bm, spec, rows):
    """Run the CPU oracle on the first `rows` rows of C; returns (seconds, flops)."""
    import oracle
    M, N, K, dtype = spec["M"], spec["N"], spec["K"], spec["dtype"]
    la, lb = spec["layout_a"], spec["layout_b"]
    Ar = A[:rows] if la == 0 else np.ascontiguousarray(A[:, :rows])
    t0 = time.perf_counter()
    oracle.gemm(Ar, Bm, rows, N, K, dtype, la, lb, with_abs=False)
    return time.perf_counter() - t0, 2.0 * rows * N * K


def cpu_baseline(A, Bm, spec, target_s=10.0):
    import oracle
    oracle.build()
    rows = 16
    secs, fl = oracle_rows_gflops(A, Bm, spec, rows)
    while secs < 1.0 and rows < spec["M"]:          # probe long enough to use every thread
        rows = min(spec["M"], rows * 4)
        secs, fl = oracle_rows_gflops(A, Bm, spec, rows)
    rows = int(min(spec["M"], max(8, rows * target_s / max(secs, 1e-3))))
    rows = max(8, rows // 8 * 8)
    secs, fl = oracle_rows_gflops(A, Bm, spec, rows)
    return {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "first %d of %d rows of C (%s), fp64 sum + one rounding, %.1f s"
                      % (rows, spec["M"], spec["name"], secs)}


def run_reference(args, spec, A, Bm):
    """The reference arm: the CPU oracle, timed per step on a bounded row sample."""
    import oracle
    oracle.build()
    rows = args.reference_rows
    for _ in range(args.warmup):
        oracle_rows_gflops(A, Bm, spec, rows)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        _, fl = oracle_rows_gflops(A, Bm, spec, rows)
        flops += fl
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = "first %d of %d rows of C (%s) per step" % (rows, spec["M"], spec["name"])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(spec, "oracle", args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "GEMM TFLOP/s (device-timed) and % of GB300 dense BF16 peak, per schedule"


L2_BYTES = 129e6


def rotation_copies(spec) -> int:
    """Copies of A, B and C to rotate so that the operands of the launches in
    flight exceed twice the L2 (1 when one copy already does)."""
    ab = 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"])
    return max(1, min(512, int(np.ceil(2 * L2_BYTES / ab)))) if ab < 2 * L2_BYTES else 1


def config_of(spec, schedule, n):
    return {"workload": spec["name"], "M": spec["M"], "N": spec["N"], "K": spec["K"],
            "dtype_in": "bf16" if spec["dtype"] == inputs.BF16 else "fp16",
            "accumulate": "fp32",
            "layout_a": "row" if spec["layout_a"] == 0 else "col",
            "layout_b": "row" if spec["layout_b"] == 0 else "col",
            "schedule": schedule, "parallelism": "replica x%d" % n,
            "l2": l2_note(spec)}


def l2_note(spec) -> str:
    ab = 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"])
    r = rotation_copies(spec)
    if r == 1:
        return "inputs %.0f MB > 2 x L2 129 MB, no flush" % (ab / 1e6)
    return "inputs %.1f MB rotated over %d copies (%.0f MB > 2 x L2 129 MB), no flush" % (
        ab / 1e6, r, r * ab / 1e6)


# --------------------------------------------------------------------- ranks
def max_over_ranks(value: float, dist, world: int, device) -> float:
    """Max of a per-rank number over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Aggregate throughput: every rank ran `steps` steps; time = slowest rank."""
    return world * steps * flops_per_step / (max_ms * 1e-3) / 1e12


def sm_busy_fraction(stamps: np.ndarray, num_sms: int) -> dict:
    """From per-CTA (start, ready, loads_done, end) stamps: the share of SM time
    occupied by CTAs between the first start and the last end, and the span."""
    start, end = stamps[:, 0].astype(np.float64), stamps[:, 3].astype(np.float64)
    span = end.max() - start.min()
    busy = float(np.sum(end - start) / (num_sms * span)) if span > 0 else 0.0
    last = np.sort(end)
    return {"sm_busy_frac": busy, "span_us": span / 1e3,
            "tail_us": float((last[-1] - np.median(last)) / 1e3)}


# --------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="square8192_bf16", choices=list(inputs.WORKLOADS))
    ap.add_argument("--schedule", default="best", choices=SCHED_NAMES + ["best"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--reference-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        spec, A, Bm = inputs.workload(args.workload)
        run_reference(args, spec, A, Bm)
        return

    import torch
    import torch.distributed as dist

    from persistent_stream_matmul_gb300 import _binding as B
    from persistent_stream_matmul_gb300 import build

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    build.build()
    B.load()

    spec, A, Bm = inputs.workload(args.workload)
    M, N, K, dtype = spec["M"], spec["N"], spec["K"], spec["dtype"]
    la, lb = spec["layout_a"], spec["layout_b"]
    flops = 2.0 * M * N * K
    alg_bytes = 2.0 * (M * K + K * N + M * N)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(Bm.view(np.int16)).cuda()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    # operands smaller than twice the L2: rotate copies so that no timed launch
    # finds its inputs left in L2 by the one before
    copies = rotation_copies(spec)
    sets = [(dA, dB, dC)] + [(dA.clone(), dB.clone(), torch.empty_like(dC))
                             for _ in range(copies - 1)]
    stream = torch.cuda.current_stream()

    plans, wss = {}, {}
    for s in SCHED_NAMES:
        sched_kind, opts = SCHED_DEFS[s]
        plans[s] = B.Plan(M, N, K, dtype, la, lb, sched_kind, **opts)
        n = plans[s].workspace_size
        wss[s] = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(device_pci_id(torch, local_rank))
    sampler.start()

    # per-schedule device time (each launch bracketed by events on this stream),
    # in interleaved rounds so that every schedule samples the same drift of
    # the clocks under the power cap
    per_sched = {}
    names = SCHED_NAMES if args.schedule == "best" else [args.schedule]
    rounds = 3
    per_round = max(1, -(-args.steps // rounds))
    times = {s: [] for s in names}
    for rnd in range(rounds):
        for s in names:
            p, w = plans[s], wss[s]
            for i in range(args.warmup if rnd == 0 else 1):
                p.run(*sets[i % copies], w, stream)
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * per_round)]
            for i in range(per_round):
                ev[2 * i].record(stream)
                p.run(*sets[(args.warmup + i) % copies], w, stream)
                ev[2 * i + 1].record(stream)
            torch.cuda.synchronize()
            st = p.last_status(stream)
            if st != B.GEMM_OK:
                raise RuntimeError("device status after %s: %s" % (s, B.gemm_status_string(st)))
            times[s] += [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(per_round)]
    for s in names:
        p, w = plans[s], wss[s]
        ms = times[s]
        med = statistics.median(ms)
        per_sched[s] = {"tflops": flops / (med * 1e-3) / 1e12, "ms_median": med,
                        "ms_min": min(ms), "ms_max": max(ms)}
        # one more (untimed) launch with per-CTA stamps: SM idle time at the tail
        ctas = p.info("grid")
        tbuf = torch.zeros(4 * ctas, dtype=torch.int64, device="cuda")
        p.set_trace(tbuf, tbuf.numel() * 8)
        p.run(dA, dB, dC, w, stream)
        torch.cuda.synchronize()
        p.set_trace(None, 0)
        per_sched[s].update(sm_busy_fraction(tbuf.cpu().numpy().reshape(ctas, 4),
                                             p.info("num_sms")))
        per_sched[s]["ctas"] = ctas
        per_sched[s]["tile"] = "%dx%dx64" % (p.info("tile_m"), p.info("tile_n"))

    best = max(per_sched, key=lambda s: per_sched[s]["tflops"])
    sched = best if args.schedule == "best" else args.schedule
    p, w = plans[sched], wss[sched]

    # headline: exactly K steps, barrier + synchronize on both sides, max over ranks
    for i in range(args.warmup):
        p.run(*sets[i % copies], w, stream)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        p.run(*sets[(args.warmup + i) % copies], w, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = e0.elapsed_time(e1)
    if p.last_status(stream) != B.GEMM_OK:
        raise RuntimeError("device status after the timed region is not OK")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, world, "cuda")
    value = whole_job_tflops(flops, args.steps, world, elapsed_ms)
    launch_ms = elapsed_ms / args.steps

    # end to end through the C ABI with host buffers: H2D A, B; GEMM; D2H C
    e2e = None
    if not args.no_e2e:
        hA = torch.from_numpy(A.view(np.int16)).reshape(-1).pin_memory()
        hB = torch.from_numpy(Bm.view(np.int16)).reshape(-1).pin_memory()
        hC = torch.empty(M * N, dtype=torch.int16).pin_memory()
        n_e2e = max(3, min(args.steps, 20))
        for _ in range(3):
            p.run_host(hA, hB, hC, dA, dB, dC, w, stream)
        barrier()
        torch.cuda.synchronize()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n_e2e):
            p.run_host(hA, hB, hC, dA, dB, dC, w, stream)
        e3.record(stream)
        torch.cuda.synchronize()
        barrier()
        te = max_over_ranks(e2.elapsed_time(e3), dist, world, "cuda")
        e2e = {"value": whole_job_tflops(flops, n_e2e, world, te),
               "unit": "TFLOP/s", "steps": n_e2e,
               "h2d_bytes_per_step": int(hA.numel() * 2 + hB.numel() * 2),
               "d2h_bytes_per_step": int(hC.numel() * 2),
               "host_chunks": p.info("host_chunks")}

    clocks = sampler.stop()

    if rank != 0:
        dist.destroy_process_group() if world > 1 else None
        return

    pk, pk_src = peaks()
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    bound = "tensor" if flops / alg_bytes >= ridge else "hbm"
    if bound == "tensor":
        achieved = flops / (launch_ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"]       # fp16 and bf16 share the dense tensor rate
        unit = "TFLOP/s"
    else:
        achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        unit = "GB/s"
    traffic = profiled_traffic(spec["name"], resolved_name(sched, p))
    for s in per_sched:
        per_sched[s]["frac_of_%s_peak" % pk_src] = (
            per_sched[s]["tflops"] / pk["bf16_tflops"] if bound == "tensor"
            else alg_bytes / (per_sched[s]["ms_median"] * 1e-3) / 1e9 / pk["hbm_gbs"])

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if dtype == inputs.BF16 else "fp16", "data": "synthetic",
        "config": config_of(spec, sched, world),
        "per_schedule": per_sched,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "peak_source": pk_src + " (burst)",
                     "traffic": traffic, "algorithmic_bytes": alg_bytes,
                     "kernel": "psm::gemm_kernel"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(A, Bm, spec)
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
