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
