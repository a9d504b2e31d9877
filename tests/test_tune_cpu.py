"""Host logic of the tuning sweeps (no GPU)."""
import math

from persistent_stream_matmul_gb300 import tune


def test_log_sampled_values_match_the_recipe():
    v = tune.log_sampled_values()
    assert v[0] == 256 and v[-1] == 8192
    assert all(x % 256 == 0 for x in v) and v == sorted(set(v))
    # spacing is logarithmic: small values are dense, large ones are every multiple
    assert 512 in v and 8192 - 256 in v
    assert len(v) == 32   # every multiple of 256 up to 8192 is hit by 1000 log-spaced points


def test_sample_shapes_is_seeded_and_bounded():
    a = tune.sample_shapes(20, seed=123, max_macs=2.0 ** 33)
    b = tune.sample_shapes(20, seed=123, max_macs=2.0 ** 33)
    assert a == b and len(set(a)) == 20
    assert all(m * n * k <= 2.0 ** 33 for m, n, k in a)
    assert tune.sample_shapes(20, seed=124, max_macs=2.0 ** 33) != a


def test_summary_ratios():
    rows = [{"M": 1, "N": 1, "K": 1, "results": {"x": {"tflops": 2.0}, "y": {"tflops": 1.0}}},
            {"M": 1, "N": 1, "K": 1, "results": {"x": {"tflops": 1.0}, "y": {"tflops": 4.0}}}]
    s = tune.summarize_shapes(rows)
    assert math.isclose(s["x"]["geomean_vs_best"], math.sqrt(1.0 * 0.25))
    assert s["x"]["wins"] == 1 and s["y"]["wins"] == 1


def test_paired_compare_alternates_and_reports_the_paired_ratio(monkeypatch):
    calls = []

    class FakeOps:
        def __init__(self, M, N, K, torch_mod):
            self.M, self.N, self.K = M, N, K

    def fake_burst(ops, dtype, la, lb, schedule, options, launches):
        calls.append((schedule, dict(options), launches))
        return 90.0 if schedule == "streamk" else 100.0     # the variant is 10 % faster

    monkeypatch.setattr(tune, "Operands", FakeOps)
    monkeypatch.setattr(tune, "burst_us", fake_burst)
    r = tune.paired_compare(8192, 8192, 8192, {"schedule": "persistent", "group_m": 8},
                            {"schedule": "streamk"}, pairs=4, torch_mod=object())
    assert math.isclose(r["variant_over_base_pct"], -10.0)
    assert r["variant_faster_pairs"] == 4 and r["pairs"] == 4
    assert r["base"] == {"schedule": "persistent", "group_m": 8}   # the caller's dicts are untouched
    timed = [c[0] for c in calls[1:]]                               # after the sizing burst
    assert timed == ["persistent", "streamk", "streamk", "persistent"] * 2
    assert all(c[1] == {"group_m": 8} for c in calls if c[0] == "persistent")
    assert r["launches"] == int(20.0 * 1e3 / 100.0)


def test_markdown_tables_and_auto_choice():
    rows = [{"M": 64, "N": 8192, "K": 8192, "results": {
                "streamk": {"tflops": 260.0}, "splitk_cluster": {"tflops": 300.0},
                "auto": {"tflops": 299.0, "schedule": 3, "split_k_cluster": 1, "sk_mode": 0}}},
            {"M": 8192, "N": 8192, "K": 8192, "results": {
                "streamk": {"tflops": 1600.0}, "splitk_cluster": {"refused": "x"},
                "auto": {"tflops": 1600.0, "schedule": 2, "split_k_cluster": 0, "sk_mode": 1}}}]
    md = tune.markdown(rows, "t")
    assert "| 64 | 8192 | 8192 | 260.0 | **300.0** | 299.0 (splitk_cluster) | 0.997 |" in md
    assert "| 8192 | 8192 | 8192 | **1600.0** | - | 1600.0 (streamk_all) | 1.000 |" in md
    assert "- auto:" in md
    g = tune.grid_markdown([{"M": 1, "N": 2, "K": 3, "grid": 152, "two_tiles": 1, "us": 10.0, "tflops": 1.5},
                            {"M": 1, "N": 2, "K": 3, "grid": 300, "two_tiles": 0, "refused": "no"}])
    assert "| 152 | 1 | 10.0 | 1.5 |" in g and "| 300 | 0 | refused | - |" in g
    assert len(tune.SKINNY_SHAPES) == 45 and all(m <= 128 for m, _, _ in tune.SKINNY_SHAPES)
