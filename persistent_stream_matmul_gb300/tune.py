"""Timing sweeps over plan options (device-timed, CUDA events).

* ``grid_sweep``: the Stream-K grid sweep of the GitHub issue "Stream-k matmul
  implementation very slow ..." (final version, log-sampled benchmark): for
  each shape, g in {#SM, 2 x #SM, #tiles when below 2 x #SM, ten random even
  values below 2 x #SM}, each with and without the two_tiles rule.  Grids
  whose CTAs cannot all be resident at once (more than one CTA per SM) are
  reported as refused: the owners of split tiles wait on their peers.
* ``shape_sweep``: the same issue's shape sampler: M, N and K drawn from
  multiples of 256 spaced evenly in log2 between 256 and 8192, a fixed random
  sample of the triples (seed 123); each shape timed with every schedule and
  with GEMM_SCHED_AUTO.  ``--large`` adds ``LARGE_SHAPES``, products of four or
  more waves of tiles that the sampler rarely draws under its size cap; the
  rule for that regime in GEMM_SCHED_AUTO was fitted on them.  ``--skinny``
  times ``SKINNY_SHAPES`` (one row of 128-row tiles, fp16, row-major A and B,
  the type and layouts of the skinny workload), on which AUTO's choice of
  cluster split-K for single-row products was fitted.
* ``--out`` keeps every record as JSON lines and ``--markdown`` renders them
  as tables (per shape: each variant's TFLOP/s, what AUTO ran and its ratio to
  the best variant; per variant: the geometric mean of its ratio to the best).

* ``paired_compare``: two option sets (or schedules) on one shape, timed in
  short bursts that alternate between them (the order flips every pair), so
  both see the same drift of the clocks under the power cap; reports the
  median ratio and how many pairs each side won.
* ``vs_cublas``: one plan against torch.matmul (cuBLAS) on the same bf16
  operands, in ~100 ms bursts that alternate, with the plan's SM clock and
  its launch time in SM cycles (the clock settles lower for a kernel that
  draws more power, so cycles compare kernel efficiency and microseconds
  compare throughput under the cap).  ``--cublas-only`` runs the cuBLAS
  launches alone, for a profiler capture of the vendor kernel.

Run as ``python -m persistent_stream_matmul_gb300.tune --help``.  Operands
are random device data (timing does not depend on the values); correctness
over sampled shapes is checked by the test suite, not here.
"""
from __future__ import annotations

import argparse
import json
import math
import random
import statistics

from . import _binding as B

SCHEDULE_VARIANTS = {
    "dp": ("dp", {}),
    "persistent": ("persistent", {}),
    "streamk": ("streamk", {}),
    "streamk_all": ("streamk", {"sk_mode": 1}),
    "splitk": ("splitk", {}),
    "splitk_cluster": ("splitk", {"split_cluster": 1}),
    "auto": ("auto", {}),
}


# four or more waves of 256 x 256 tiles on 76 SM pairs, short and long k
LARGE_SHAPES = [(8192, 8192, 8192), (8192, 14336, 4096), (4096, 4096, 4096), (16384, 4096, 4096),
                (6144, 6144, 6144), (8192, 4096, 8192), (4096, 14336, 4096), (2048, 8192, 8192),
                (3072, 3072, 8192), (12288, 12288, 2048), (4096, 8192, 2048), (8192, 8192, 1024),
                (5120, 5120, 5120), (2560, 10240, 4096)]


# one row of 128-row tiles: skinny, memory-bound products
SKINNY_SHAPES = [(m, n, k) for m in (16, 64, 128) for n in (1024, 2048, 4096, 8192, 16384)
                 for k in (1024, 4096, 16384)]


def log_sampled_values(lo: int = 256, hi: int = 8192, step: int = 256, n: int = 1000):
    """Multiples of `step` spaced evenly in log2 between lo and hi, deduplicated."""
    a, b = math.log2(lo), math.log2(hi)
    vals = {int(round(2 ** (a + (b - a) * i / (n - 1)) / step)) * step for i in range(n)}
    return sorted(v for v in vals if v > 0)


def sample_shapes(count: int, seed: int = 123, max_macs: float | None = None):
    """`count` (M, N, K) triples sampled without replacement from all triples."""
    vals = log_sampled_values()
    triples = [(m, n, k) for m in vals for n in vals for k in vals]
    if max_macs:
        triples = [t for t in triples if t[0] * t[1] * t[2] <= max_macs]
    return random.Random(seed).sample(triples, count)


class Operands:
    """Random bf16/fp16 device operands, reused across plans of one shape."""

    def __init__(self, M, N, K, torch_mod):
        t = torch_mod
        self.M, self.N, self.K = M, N, K
        self.a = t.randn(M * K, device="cuda").to(t.bfloat16).view(t.int16)
        self.b = t.randn(K * N, device="cuda").to(t.bfloat16).view(t.int16)
        self.c = t.empty(M * N, dtype=t.int16, device="cuda")
        self.t = t
        self.ws = None

    def workspace(self, nbytes):
        if nbytes == 0:
            return None
        if self.ws is None or self.ws.numel() < nbytes:
            self.ws = self.t.zeros(nbytes, dtype=self.t.uint8, device="cuda")
        return self.ws


def time_plan(ops: Operands, dtype, la, lb, schedule, options, warmup=3, iters=10):
    """Median device time (us) of one gemm_run, or a refusal reason."""
    t = ops.t
    try:
        p = B.Plan(ops.M, ops.N, ops.K, dtype, la, lb, schedule, **options)
    except B.GemmError as e:
        return {"refused": str(e)}
    try:
        w = ops.workspace(p.workspace_size)
        stream = t.cuda.current_stream()
        for _ in range(warmup):
            p.run(ops.a, ops.b, ops.c, w, stream)
        ev = [t.cuda.Event(enable_timing=True) for _ in range(2 * iters)]
        for i in range(iters):
            ev[2 * i].record(stream)
            p.run(ops.a, ops.b, ops.c, w, stream)
            ev[2 * i + 1].record(stream)
        t.cuda.synchronize()
        st = p.last_status(stream)
        if st != B.GEMM_OK:
            return {"refused": B.gemm_status_string(st)}
        us = statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(iters)) * 1e3
        flops = 2.0 * ops.M * ops.N * ops.K
        return {"us": us, "tflops": flops / (us * 1e-6) / 1e12,
                "schedule": p.info("schedule"), "sk_mode": p.info("sk_mode"),
                "split_k_cluster": p.info("split_k_cluster"),
                "tile": "%dx%d" % (p.info("tile_m"), p.info("tile_n")), "grid": p.info("grid")}
    except B.GemmError as e:
        return {"refused": str(e)}
    finally:
        p.close()


def burst_us(ops: Operands, dtype, la, lb, schedule, options, launches):
    """Mean device time (us) of `launches` back-to-back runs of one plan."""
    t = ops.t
    p = B.Plan(ops.M, ops.N, ops.K, dtype, la, lb, schedule, **options)
    try:
        w = ops.workspace(p.workspace_size)
        stream = t.cuda.current_stream()
        for _ in range(3):
            p.run(ops.a, ops.b, ops.c, w, stream)
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(launches):
            p.run(ops.a, ops.b, ops.c, w, stream)
        e1.record(stream)
        t.cuda.synchronize()
        if p.last_status(stream) != B.GEMM_OK:
            raise B.GemmError(p.last_status(stream), "paired_compare")
        return e0.elapsed_time(e1) / launches * 1e3
    finally:
        p.close()


def paired_compare(M, N, K, base, variant, dtype=B.GEMM_BF16, la=0, lb=1, pairs=10,
                   burst_ms=20.0, torch_mod=None):
    """`base` and `variant` are dicts of plan options plus an optional
    "schedule" (default "streamk"); returns medians and the paired ratio."""
    import torch as t
    t = torch_mod or t
    ops = Operands(M, N, K, t)
    sides = {"base": dict(base), "variant": dict(variant)}
    scheds = {k: v.pop("schedule", "streamk") for k, v in sides.items()}
    # launches per burst from one timing of the base
    one = burst_us(ops, dtype, la, lb, scheds["base"], sides["base"], 3)
    launches = max(5, int(burst_ms * 1e3 / max(one, 1.0)))
    times = {"base": [], "variant": []}
    for i in range(pairs):
        order = ("base", "variant") if i % 2 == 0 else ("variant", "base")
        for side in order:
            times[side].append(burst_us(ops, dtype, la, lb, scheds[side], sides[side], launches))
    ratios = [v / b for b, v in zip(times["base"], times["variant"])]
    return {"M": M, "N": N, "K": K, "base": base, "variant": variant, "launches": launches,
            "base_us": statistics.median(times["base"]),
            "variant_us": statistics.median(times["variant"]),
            "variant_over_base_pct": 100.0 * (statistics.median(ratios) - 1.0),
            "variant_faster_pairs": sum(1 for r in ratios if r < 1.0), "pairs": pairs}


def vs_cublas(M, N, K, schedule="streamk", options=None, rounds=6, burst_ms=100.0, torch_mod=None):
    """Long bursts of one plan and of torch.matmul (cuBLAS) on the same bf16
    operands (A row-major, B column-major), alternating, the order flipping
    every round.  Each burst lasts about `burst_ms`, long enough for the clocks
    to settle under the power cap for that kernel; the median launch of its
    last two thirds is kept.  The plan's launches also carry per-CTA stamps,
    so its SM clock (%clock64 over %globaltimer) and its launch time in SM
    cycles are reported beside the times."""
    import numpy as np
    import torch as t
    t = torch_mod or t
    a = t.randn(M, K, device="cuda").to(t.bfloat16)
    bt = t.randn(N, K, device="cuda").to(t.bfloat16)  # B column-major: its transpose, row-major
    c = t.empty(M, N, dtype=t.bfloat16, device="cuda")
    p = B.Plan(M, N, K, B.GEMM_BF16, 0, 1, schedule, **(options or {}))
    w = t.zeros(max(1, p.workspace_size), dtype=t.uint8, device="cuda")
    ctas = p.info("grid")
    stamps = t.zeros(ctas * B.TRACE_STAMPS, dtype=t.int64, device="cuda")
    p.set_trace(stamps, stamps.numel() * 8)
    stream = t.cuda.current_stream()
    flops = 2.0 * M * N * K
    arms = {"library": lambda: p.run(a, bt, c, w if p.workspace_size else None, stream),
            "cublas": lambda: t.matmul(a, bt.t(), out=c)}
    n = max(20, int(burst_ms * 1e3 / (flops / 1.6e15 * 1e6)))

    def burst(fn):
        ev = [t.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        t.cuda.synchronize()
        ev[0].record(stream)
        for i in range(n):
            fn()
            ev[i + 1].record(stream)
        t.cuda.synchronize()
        d = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(n)]
        return statistics.median(d[n // 3:])

    times = {"library": [], "cublas": []}
    mhz = []
    for r in range(rounds):
        for arm in (("library", "cublas") if r % 2 == 0 else ("cublas", "library")):
            times[arm].append(burst(arms[arm]))
            if arm == "library":
                s = stamps.cpu().numpy().reshape(ctas, B.TRACE_STAMPS).astype(np.float64)
                ns, cyc = s[:, 3] - s[:, 0], s[:, 5] - s[:, 4]
                mhz.append(float(np.median(cyc[ns > 0] / ns[ns > 0])) * 1e3)
    p.set_trace(None, 0)
    assert p.last_status(stream) == B.GEMM_OK
    p.close()
    lib_us, cub_us = statistics.median(times["library"]), statistics.median(times["cublas"])
    sm_mhz = statistics.median(mhz)
    return {"M": M, "N": N, "K": K, "schedule": schedule, "options": options or {},
            "launches_per_burst": n, "rounds": rounds,
            "library_us": lib_us, "cublas_us": cub_us,
            "library_tflops": flops / lib_us / 1e6, "cublas_tflops": flops / cub_us / 1e6,
            "library_over_cublas": statistics.median(
                [cb / lb for lb, cb in zip(times["library"], times["cublas"])]),
            "library_sm_mhz": sm_mhz, "library_kcycles": lib_us * sm_mhz / 1e3}


def cublas_only(M, N, K, launches=8, torch_mod=None):
    """torch.matmul (cuBLAS) launches alone on the operands `vs_cublas` uses,
    for a profiler capture of the vendor kernel."""
    import torch as t
    t = torch_mod or t
    a = t.randn(M, K, device="cuda").to(t.bfloat16)
    bt = t.randn(N, K, device="cuda").to(t.bfloat16)
    c = t.empty(M, N, dtype=t.bfloat16, device="cuda")
    for _ in range(launches):
        t.matmul(a, bt.t(), out=c)
    t.cuda.synchronize()


def grid_sweep(M, N, K, dtype=B.GEMM_BF16, la=0, lb=1, seed=123, torch_mod=None):
    import torch as t
    t = torch_mod or t
    sms = t.cuda.get_device_properties(0).multi_processor_count
    probe = B.Plan(M, N, K, dtype, la, lb, "streamk")
    tiles = probe.info("tiles") * probe.info("cluster_m")
    probe.close()
    grids = [sms, 2 * sms] + ([tiles] if tiles < 2 * sms else [])
    grids += random.Random(seed).sample(range(2, 2 * sms, 2), 10)
    ops = Operands(M, N, K, t)
    rows = []
    for two in (1, 0):
        for g in grids:
            r = time_plan(ops, dtype, la, lb, "streamk", {"grid": g, "two_tiles": two})
            rows.append({"M": M, "N": N, "K": K, "grid": g, "two_tiles": two, **r})
    return rows


def shape_sweep(count, dtype=B.GEMM_BF16, la=0, lb=1, seed=123, max_macs=2.0 ** 36,
                variants=None, torch_mod=None, extra_shapes=()):
    import torch as t
    t = torch_mod or t
    variants = variants or list(SCHEDULE_VARIANTS)
    rows = []
    shapes = list(sample_shapes(count, seed, max_macs)) if count else []
    for (M, N, K) in shapes + list(extra_shapes):
        ops = Operands(M, N, K, t)
        res = {}
        for name in variants:
            sched, opt = SCHEDULE_VARIANTS[name]
            res[name] = time_plan(ops, dtype, la, lb, sched, opt)
        rows.append({"M": M, "N": N, "K": K, "dtype": "bf16" if dtype == B.GEMM_BF16 else "fp16",
                     "layout_a": la, "layout_b": lb, "results": res})
        del ops
    return rows


def auto_runs(r: dict) -> str:
    """The variant name of what AUTO resolved to, from its timing record."""
    kind = {0: "dp", 1: "persistent", 2: "streamk", 3: "splitk"}.get(r.get("schedule"), "?")
    if kind == "splitk" and r.get("split_k_cluster"):
        return "splitk_cluster"
    if kind == "streamk" and r.get("sk_mode"):
        return "streamk_all"
    return kind


def markdown(rows, title: str) -> str:
    """A shape sweep as a table: TFLOP/s per variant, AUTO's choice and its
    ratio to the best variant, then the geometric means of summarize_shapes."""
    if not rows:
        return ""
    names = [n for n in rows[0]["results"] if n != "auto"]
    out = ["## " + title, "",
           "| M | N | K | " + " | ".join(names) + " | auto (runs) | auto / best |",
           "|---:|---:|---:|" + "---:|" * len(names) + "---|---:|"]
    for r in rows:
        res = r["results"]
        best = max(v.get("tflops", 0.0) for v in res.values())
        cells = []
        for n in names:
            v = res[n].get("tflops")
            cells.append(("**%.1f**" if v == best else "%.1f") % v if v else "-")
        a = res.get("auto", {})
        cells.append("%.1f (%s)" % (a["tflops"], auto_runs(a)) if a.get("tflops") else "-")
        cells.append("%.3f" % (a["tflops"] / best) if a.get("tflops") and best else "-")
        out.append("| %d | %d | %d | " % (r["M"], r["N"], r["K"]) + " | ".join(cells) + " |")
    out += ["", "Geometric mean of each variant's TFLOP/s over the best variant of the shape:", ""]
    for n, v in summarize_shapes(rows).items():
        out.append("- %s: %.4f (best on %d of %d shapes)" % (n, v["geomean_vs_best"], v["wins"], v["shapes"]))
    return "\n".join(out) + "\n"


def grid_markdown(rows) -> str:
    if not rows:
        return ""
    r0 = rows[0]
    out = ["## Stream-K grid sweep, %d x %d x %d" % (r0["M"], r0["N"], r0["K"]), "",
           "| grid (CTAs) | two_tiles | us | TFLOP/s |", "|---:|---:|---:|---:|"]
    for r in sorted(rows, key=lambda r: (-r["two_tiles"], r["grid"])):
        if "us" in r:
            out.append("| %d | %d | %.1f | %.1f |" % (r["grid"], r["two_tiles"], r["us"], r["tflops"]))
        else:
            out.append("| %d | %d | refused | - |" % (r["grid"], r["two_tiles"]))
    return "\n".join(out) + "\n"


def summarize_shapes(rows):
    """Geometric-mean throughput ratios of each variant to the best per shape."""
    names = list(rows[0]["results"]) if rows else []
    out = {}
    for n in names:
        ratios = []
        for r in rows:
            best = max(v.get("tflops", 0.0) for v in r["results"].values())
            v = r["results"][n].get("tflops")
            if v and best:
                ratios.append(v / best)
        if ratios:
            out[n] = {"geomean_vs_best": math.exp(sum(math.log(x) for x in ratios) / len(ratios)),
                      "wins": sum(1 for r in rows if max(r["results"], key=lambda k:
                                  r["results"][k].get("tflops", 0.0)) == n),
                      "shapes": len(ratios)}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--grid-sweep", nargs=3, type=int, metavar=("M", "N", "K"))
    ap.add_argument("--shapes", type=int, default=0, help="log-sampled shapes to time")
    ap.add_argument("--max-macs", type=float, default=2.0 ** 36)
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16")
    ap.add_argument("--large", action="store_true", help="also time LARGE_SHAPES")
    ap.add_argument("--compare", nargs=5, metavar=("M", "N", "K", "BASE", "VARIANT"),
                    help="paired bursts; BASE and VARIANT are JSON option dicts, e.g. "
                         "'{\"schedule\": \"persistent\"}' '{\"schedule\": \"streamk\"}'")
    ap.add_argument("--layout-b", type=int, default=1, help="0 row-major, 1 column-major B")
    ap.add_argument("--skinny", action="store_true",
                    help="time SKINNY_SHAPES (fp16, row-major A and B)")
    ap.add_argument("--vs-cublas", nargs=3, type=int, metavar=("M", "N", "K"),
                    help="bf16 plan (--schedule) against torch.matmul in long alternating bursts")
    ap.add_argument("--schedule", default="streamk", help="schedule for --vs-cublas")
    ap.add_argument("--cublas-only", nargs=3, type=int, metavar=("M", "N", "K"),
                    help="eight torch.matmul launches alone (for a profiler capture)")
    ap.add_argument("--out", help="also write every record to this file as JSON lines")
    ap.add_argument("--markdown", help="write the sweeps as markdown tables to this file")
    args = ap.parse_args()
    dtype = B.GEMM_BF16 if args.dtype == "bf16" else B.GEMM_F16
    if args.cublas_only:
        cublas_only(*args.cublas_only)
        return
    B.load()
    if args.vs_cublas:
        print(json.dumps(vs_cublas(*args.vs_cublas, schedule=args.schedule)), flush=True)
    if args.compare:
        M, N, K = (int(x) for x in args.compare[:3])
        print(json.dumps(paired_compare(M, N, K, json.loads(args.compare[3]), json.loads(args.compare[4]),
                                        dtype=dtype, lb=args.layout_b)), flush=True)
    records, md = [], []

    def emit(rec):
        records.append(rec)
        print(json.dumps(rec), flush=True)

    if args.grid_sweep:
        rows = grid_sweep(*args.grid_sweep, dtype=dtype)
        for row in rows:
            emit(row)
        md.append(grid_markdown(rows))
    if args.shapes or args.large:
        rows = shape_sweep(args.shapes, dtype=dtype, max_macs=args.max_macs, lb=args.layout_b,
                           extra_shapes=LARGE_SHAPES if args.large else ())
        for row in rows:
            emit(row)
        emit({"summary": summarize_shapes(rows)})
        md.append(markdown(rows, "Log-sampled and large shapes, %s, A row-major, B %s-major"
                           % (args.dtype, "column" if args.layout_b else "row")))
    if args.skinny:
        rows = shape_sweep(0, dtype=B.GEMM_F16, la=0, lb=0, extra_shapes=SKINNY_SHAPES)
        for row in rows:
            emit(row)
        emit({"summary_skinny": summarize_shapes(rows)})
        md.append(markdown(rows, "Single row of tiles (skinny), fp16, A and B row-major"))
    if args.out:
        with open(args.out, "w") as f:
            for rec in records:
                f.write(json.dumps(rec) + "\n")
    if args.markdown:
        with open(args.markdown, "w") as f:
            f.write("\n".join(m for m in md if m))


if __name__ == "__main__":
    main()
