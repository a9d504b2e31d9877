#!/usr/bin/env python3
"""Benchmark: GEMM TFLOP/s (device-timed) and fraction of the GB300 roofline,
per schedule, on the five synthetic workloads.

The headline workload (default: bf16 8192 x 8192 x 8192, row-major A,
column-major B) gives the line's ``value``: K back-to-back steps of one
C = A*B through the C ABI (gemm_run), with the schedule that measured fastest
per launch.  The four other workloads get the same measurement under
``per_workload`` (every schedule's per-launch median, the best schedule back
to back, the roofline fraction: tensor, or HBM for the memory-bound skinny
product).  Prints one JSON line.

  python bench.py [--steps K] [--warmup W] [--workload NAME]
                  [--schedule dp|persistent|streamk|...|best] [--impl ours|reference]
                  [--only-headline]

The library issues cluster-multicast tensor copies from this GPU's own
memory, so it runs on one GPU per process and is never part of a multi-GPU
job: with --gpus > 1 or WORLD_SIZE > 1 this arm exits with an error before
touching CUDA.

--impl reference times the CPU oracle (the plain fp64 product) on the host
cores instead, on a bounded row sample of the headline workload per step;
under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import datetime
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
SCHED_NAMES = ["dp", "persistent", "streamk", "streamk_all", "splitk", "splitk_cluster", "auto"]
# name -> (schedule, options): "streamk" is the hybrid rule of the issue's final
# version; "streamk_all" puts every tile in the Stream-K wave; "splitk_cluster"
# reduces each tile's split-K parts inside a thread-block cluster
SCHED_DEFS = {"dp": ("dp", {}), "persistent": ("persistent", {}),
              "streamk": ("streamk", {}), "streamk_all": ("streamk", {"sk_mode": 1}),
              "splitk": ("splitk", {}), "splitk_cluster": ("splitk", {"split_cluster": 1}),
              "auto": ("auto", {})}
HEADLINE = "square8192_bf16"
METRIC = "GEMM TFLOP/s (device-timed) and % of GB300 dense BF16 peak, per schedule"


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
    if kind == "splitk" and plan.info("split_k_cluster") == 1:
        return "splitk_cluster"
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
    """nvidia-smi samples every 100 ms, with their timestamps, so that the
    clocks of each measured phase can be told apart afterwards."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_id: str | None):
        self.proc = None
        self.device_id = device_id
        self.samples = []
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

    @staticmethod
    def now() -> float:
        """Local wall time in seconds, on the clock of nvidia-smi's timestamps."""
        return datetime.datetime.now().timestamp()

    @staticmethod
    def parse(lines):
        """[(t, sm_mhz, sm_max_mhz, power_w, {active reasons})] from the CSV."""
        out = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax, pw = float(parts[2]), float(parts[3]), float(parts[4])
            except ValueError:
                continue
            reasons = {n for n, v in zip(ClockSampler.REASONS, parts[6:10])
                       if v.lower().startswith("active")}
            out.append((t, sm, smax, pw, reasons))
        return out

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            self.samples = self.parse(f)
        try:
            os.unlink(self.path)
        except OSError:
            pass

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock under load, the maximum clock and the throttle
        reasons seen, over all samples or those between t0 and t1."""
        s = [x for x in self.samples if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        if not s and t0 is not None and t1 is not None:
            # a window shorter than the sampling period: the samples just around it
            s = [x for x in self.samples if t0 - 0.15 <= x[0] <= t1 + 0.15]
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        pmax = max(x[3] for x in self.samples)
        busy = [x[1] for x in s if x[3] > 0.5 * pmax] or [x[1] for x in s]
        reasons = sorted(set().union(*(x[4] for x in s)))
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(x[2] for x in s),
                "reasons": reasons, "samples": len(s), "power_w_max": max(x[3] for x in s)}


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
        "config": config_of(spec, "oracle"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def rotation_copies(spec) -> int:
    """Copies of A, B and C to rotate so that the operands of the launches in
    flight exceed twice the L2 (1 when one copy already does)."""
    ab = 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"])
    return max(1, min(512, int(np.ceil(2 * L2_BYTES / ab)))) if ab < 2 * L2_BYTES else 1


def config_of(spec, schedule):
    return {"workload": spec["name"], "M": spec["M"], "N": spec["N"], "K": spec["K"],
            "dtype_in": "bf16" if spec["dtype"] == inputs.BF16 else "fp16",
            "accumulate": "fp32",
            "layout_a": "row" if spec["layout_a"] == 0 else "col",
            "layout_b": "row" if spec["layout_b"] == 0 else "col",
            "schedule": schedule, "parallelism": "one GPU",
            "l2": l2_note(spec)}


def l2_note(spec) -> str:
    ab = 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"])
    r = rotation_copies(spec)
    if r == 1:
        return "inputs %.0f MB > 2 x L2 129 MB, no flush" % (ab / 1e6)
    return "inputs %.1f MB rotated over %d copies (%.0f MB > 2 x L2 129 MB), no flush" % (
        ab / 1e6, r, r * ab / 1e6)


def multi_gpu_request(args, env) -> str | None:
    """Why this arm refuses to run, or None: the library issues
    cluster-multicast copies, so it stays on single-GPU runs."""
    world = int(env.get("WORLD_SIZE", "1") or "1")
    if args.gpus > 1 or world > 1:
        return ("bench.py runs on one GPU only (--gpus %d, WORLD_SIZE %d): the library's "
                "kernels use cluster-multicast tensor copies and are never run by a "
                "multi-GPU job" % (args.gpus, world))
    return None


def sm_busy_fraction(stamps: np.ndarray, num_sms: int) -> dict:
    """From per-CTA (start, ready, loads_done, end) stamps: the share of SM time
    occupied by CTAs between the first start and the last end, and the span."""
    start, end = stamps[:, 0].astype(np.float64), stamps[:, 3].astype(np.float64)
    span = end.max() - start.min()
    busy = float(np.sum(end - start) / (num_sms * span)) if span > 0 else 0.0
    last = np.sort(end)
    return {"sm_busy_frac": busy, "span_us": span / 1e3,
            "tail_us": float((last[-1] - np.median(last)) / 1e3)}


def burst_sm_mhz(stamps: np.ndarray) -> list:
    """Per launch: the median over CTAs of the SM clock each CTA ran at,
    %clock64 cycles over %globaltimer nanoseconds (stamps: launches x CTAs x
    (start, ready, loads done, end, clock at start, clock at end))."""
    ns = stamps[:, :, 3].astype(np.float64) - stamps[:, :, 0]
    cyc = stamps[:, :, 5].astype(np.float64) - stamps[:, :, 4]
    with np.errstate(divide="ignore", invalid="ignore"):
        ghz = np.where(ns > 0, cyc / ns, np.nan)
    return [float(np.nanmedian(g)) * 1e3 for g in ghz]


def host_link(torch, nbytes: int = 256 << 20):
    """Pinned host <-> device copy bandwidth (GB/s, best of three) and the
    NUMA placement of the GPU and of this process's CPUs: the end-to-end
    number is bound by this link, which differs between boxes."""
    out = {}
    h = torch.empty(nbytes // 2, dtype=torch.int16).pin_memory()
    d = torch.empty_like(h, device="cuda")
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        out[name] = best
    try:
        bus = device_pci_id(torch, 0)
        with open("/sys/bus/pci/devices/%s/numa_node" % bus.lower()[4:]) as f:
            out["gpu_numa_node"] = int(f.read().strip())
    except Exception:
        out["gpu_numa_node"] = None
    try:
        cpus = os.sched_getaffinity(0)
        nodes = set()
        for n in os.listdir("/sys/devices/system/node"):
            if n.startswith("node") and n[4:].isdigit():
                with open("/sys/devices/system/node/%s/cpulist" % n) as f:
                    if cpus & parse_cpulist(f.read()):
                        nodes.add(int(n[4:]))
        out["cpu_numa_nodes"] = sorted(nodes)
        out["cpus"] = len(cpus)
    except Exception:
        out["cpu_numa_nodes"] = None
    return out


def parse_cpulist(text: str) -> set:
    """'0-3,8,10-11' -> {0, 1, 2, 3, 8, 10, 11}"""
    out = set()
    for part in text.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        out.update(range(int(a), int(b or a) + 1))
    return out


def roofline_of(spec, ms: float, pk: dict):
    """(bound, achieved, peak, unit) of one launch taking `ms` milliseconds:
    tensor-bound products are rated in TFLOP/s against the bf16 dense peak
    (fp16 has the same rate), memory-bound ones in GB/s of algorithmic bytes
    2(MK + KN + MN) against the measured HBM copy bandwidth."""
    M, N, K = spec["M"], spec["N"], spec["K"]
    flops = 2.0 * M * N * K
    alg_bytes = 2.0 * (M * K + K * N + M * N)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if flops / alg_bytes >= ridge:
        return "tensor", flops / (ms * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s"
    return "hbm", alg_bytes / (ms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s"


# --------------------------------------------------------------------- GPU arm
def measure_workload(name, args, torch, B, sampler, pk, pk_src, headline):
    """Per-schedule per-launch medians and the best (or chosen) schedule back
    to back on one workload; for the headline also end to end."""
    spec, A, Bm = inputs.workload(name)
    M, N, K, dtype = spec["M"], spec["N"], spec["K"], spec["dtype"]
    la, lb = spec["layout_a"], spec["layout_b"]
    flops = 2.0 * M * N * K
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(Bm.view(np.int16)).cuda()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    # operands smaller than twice the L2: rotate copies so that no timed launch
    # finds its inputs left in L2 by the one before
    copies = rotation_copies(spec)
    sets = [(dA, dB, dC)] + [(dA.clone(), dB.clone(), torch.empty_like(dC))
                             for _ in range(copies - 1)]
    stream = torch.cuda.current_stream()

    chosen = args.schedule if headline else "best"
    names = SCHED_NAMES if chosen == "best" else [chosen]
    plans, wss = {}, {}
    for s in names:
        sched_kind, opts = SCHED_DEFS[s]
        plans[s] = B.Plan(M, N, K, dtype, la, lb, sched_kind, **opts)
        n = plans[s].workspace_size
        wss[s] = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None

    # per-schedule device time (each launch bracketed by events on this stream),
    # in interleaved rounds so that every schedule samples the same drift of
    # the clocks under the power cap
    per_sched = {}
    rounds = 3
    per_round = max(1, -(-args.steps // rounds))
    times = {s: [] for s in names}
    t_phase0 = sampler.now()
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
                raise RuntimeError("device status after %s on %s: %s"
                                   % (s, name, B.gemm_status_string(st)))
            times[s] += [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(per_round)]
    t_phase1 = sampler.now()
    for s in names:
        p, w = plans[s], wss[s]
        ms = times[s]
        med = statistics.median(ms)
        bound, ach, peak, unit = roofline_of(spec, med, pk)
        per_sched[s] = {"tflops": flops / (med * 1e-3) / 1e12, "ms_median": med,
                        "ms_mean": statistics.fmean(ms), "ms_min": min(ms), "ms_max": max(ms),
                        "frac_of_%s_peak" % pk_src: ach / peak}
        # one more (untimed) launch with per-CTA stamps: SM idle time at the tail
        ctas = p.info("grid")
        tbuf = torch.zeros(B.TRACE_STAMPS * ctas, dtype=torch.int64, device="cuda")
        p.set_trace(tbuf, tbuf.numel() * 8)
        p.run(dA, dB, dC, w, stream)
        torch.cuda.synchronize()
        p.set_trace(None, 0)
        per_sched[s].update(sm_busy_fraction(tbuf.cpu().numpy().reshape(ctas, B.TRACE_STAMPS),
                                             p.info("num_sms")))
        per_sched[s]["ctas"] = ctas
        per_sched[s]["tile"] = "%dx%dx64" % (p.info("tile_m"), p.info("tile_n"))
        per_sched[s]["runs"] = resolved_name(s, p)

    best = max(per_sched, key=lambda s: per_sched[s]["tflops"])
    sched = best if chosen == "best" else chosen
    p, w = plans[sched], wss[sched]

    # back to back: untimed priming (about 30 ms of the same launches, so that
    # the clocks leave whatever state the per-variant rounds, with their idle
    # gaps, left them in), the W warm-up steps, then exactly K steps with a
    # synchronize on both sides
    priming = min(2000, max(args.warmup, int(30.0 / max(per_sched[sched]["ms_median"], 1e-3))))
    for i in range(priming):
        p.run(*sets[i % copies], w, stream)
    for i in range(args.warmup):
        p.run(*sets[i % copies], w, stream)
    torch.cuda.synchronize()
    t_head0 = sampler.now()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        p.run(*sets[(args.warmup + i) % copies], w, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t_head1 = sampler.now()
    elapsed_ms = e0.elapsed_time(e1)
    if p.last_status(stream) != B.GEMM_OK:
        raise RuntimeError("device status after the timed region of %s is not OK" % name)
    launch_ms = elapsed_ms / args.steps
    bound, achieved, peak, unit = roofline_of(spec, launch_ms, pk)

    # after the timed region: the same burst again with an event between
    # launches and per-CTA stamps in every launch, to show how launch times
    # and the SM clock drift within a burst (the clock ramps after idle time
    # and settles under the power cap)
    ctas = p.info("grid")
    n_st = B.TRACE_STAMPS
    tb = torch.zeros(args.steps * n_st * ctas, dtype=torch.int64, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(args.steps):
        p.set_trace(tb.data_ptr() + i * n_st * ctas * 8, n_st * ctas * 8)
        p.run(*sets[(args.warmup + i) % copies], w, stream)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    p.set_trace(None, 0)
    burst = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    mhz = burst_sm_mhz(tb.cpu().numpy().reshape(args.steps, ctas, n_st))
    q = max(1, len(burst) // 4)
    drift = {"ms_first_quarter": statistics.fmean(burst[:q]),
             "ms_last_quarter": statistics.fmean(burst[-q:]),
             "ms_median": statistics.median(burst),
             "sm_mhz_first_quarter": statistics.fmean(mhz[:q]),
             "sm_mhz_last_quarter": statistics.fmean(mhz[-q:]),
             "sm_mhz_median": statistics.median(mhz)}

    out = {"spec": spec, "A": A, "Bm": Bm, "schedule": sched, "plan": p, "priming": priming,
           "elapsed_ms": elapsed_ms, "launch_ms": launch_ms,
           "tflops": flops / (launch_ms * 1e-3) / 1e12,
           "per_schedule": per_sched, "burst_drift": drift,
           "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                        "frac": achieved / peak},
           "phases": {"per_schedule": (t_phase0, t_phase1), "back_to_back": (t_head0, t_head1)}}

    # end to end through the C ABI with host buffers: H2D A, B; GEMM; D2H C
    if headline and not args.no_e2e:
        hA = torch.from_numpy(A.view(np.int16)).reshape(-1).pin_memory()
        hB = torch.from_numpy(Bm.view(np.int16)).reshape(-1).pin_memory()
        hC = torch.empty(M * N, dtype=torch.int16).pin_memory()
        n_e2e = max(3, min(args.steps, 20))
        for _ in range(3):
            p.run_host(hA, hB, hC, dA, dB, dC, w, stream)
        torch.cuda.synchronize()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n_e2e):
            p.run_host(hA, hB, hC, dA, dB, dC, w, stream)
        e3.record(stream)
        torch.cuda.synchronize()
        if p.last_status(stream) != B.GEMM_OK:
            raise RuntimeError("device status after the end-to-end region is not OK")
        te = e2.elapsed_time(e3)
        out["e2e"] = {"value": n_e2e * flops / (te * 1e-3) / 1e12,
                      "unit": "TFLOP/s", "steps": n_e2e,
                      "h2d_bytes_per_step": int(hA.numel() * 2 + hB.numel() * 2),
                      "d2h_bytes_per_step": int(hC.numel() * 2),
                      "host_chunks": p.info("host_chunks"),
                      "host_col_chunks": p.info("host_col_chunks"),
                      "host_link": host_link(torch)}
    for s in names:
        if s != sched:
            plans[s].close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=list(inputs.WORKLOADS))
    ap.add_argument("--schedule", default="best", choices=SCHED_NAMES + ["best"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--reference-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only-headline", action="store_true",
                    help="measure the --workload alone, without per_workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        spec, A, Bm = inputs.workload(args.workload)
        run_reference(args, spec, A, Bm)
        return

    why = multi_gpu_request(args, os.environ)
    if why:
        print(why, file=sys.stderr, flush=True)
        sys.exit(2)

    import torch

    from persistent_stream_matmul_gb300 import _binding as B
    from persistent_stream_matmul_gb300 import build

    torch.cuda.set_device(0)
    build.build()
    B.load()
    pk, pk_src = peaks()

    sampler = ClockSampler(device_pci_id(torch, 0))
    sampler.start()
    head = measure_workload(args.workload, args, torch, B, sampler, pk, pk_src, headline=True)
    others = {}
    if not args.only_headline:
        for name in inputs.WORKLOADS:
            if name == args.workload:
                continue
            r = measure_workload(name, args, torch, B, sampler, pk, pk_src, headline=False)
            r.pop("plan").close()
            r.pop("A"), r.pop("Bm")
            others[name] = r
            torch.cuda.empty_cache()
    sampler.stop()

    spec, p, sched = head["spec"], head["plan"], head["schedule"]
    clocks = sampler.summary()
    head_clk = sampler.summary(*head["phases"]["back_to_back"])
    sched_clk = sampler.summary(*head["phases"]["per_schedule"])
    traffic = profiled_traffic(spec["name"], resolved_name(sched, p))
    rf = head["roofline"]

    per_workload = {}
    for name, r in [(args.workload, head)] + list(others.items()):
        bt = sampler.summary(*r["phases"]["back_to_back"])
        per_workload[name] = {
            "config": config_of(r["spec"], r["schedule"]),
            "best_schedule": r["schedule"],
            "back_to_back_tflops": r["tflops"], "ms_per_step": r["launch_ms"],
            "priming_launches": r["priming"],
            "roofline": dict(r["roofline"], peak_source=pk_src + " (burst)",
                             traffic=profiled_traffic(name, r["per_schedule"][r["schedule"]]["runs"])),
            "sm_mhz_back_to_back": bt["sm_mhz"],
            "burst_drift": r["burst_drift"],
            "per_schedule": r["per_schedule"],
        }

    line = {
        "metric": METRIC, "value": head["tflops"], "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["launch_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if spec["dtype"] == inputs.BF16 else "fp16", "data": "synthetic",
        "config": dict(config_of(spec, sched), priming_launches=head["priming"]),
        "per_schedule": head["per_schedule"],
        "roofline": {"bound": rf["bound"], "achieved": rf["achieved"], "peak": rf["peak"],
                     "unit": rf["unit"], "frac": rf["frac"], "peak_source": pk_src + " (burst)",
                     "traffic": traffic,
                     "algorithmic_bytes": 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"]
                                                 + spec["M"] * spec["N"]),
                     "kernel": "psm::gemm_kernel"},
        "gpu_launches": args.steps,
        "clocks": dict(clocks, back_to_back=head_clk, per_schedule_rounds=sched_clk,
                       headline_ms_x_sm_mhz=(head["launch_ms"] * head_clk["sm_mhz"]
                                             if head_clk["sm_mhz"] else None)),
        "e2e": head.get("e2e"),
        "per_workload": per_workload,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(head["A"], head["Bm"], spec)
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
