"""Host logic of bench.py that needs no GPU: operand rotation against the L2,
the name a plan's traffic is filed under, and the hash-gated traffic lookup."""
import bench
from persistent_stream_matmul_gb300 import inputs


def _spec(name):
    M, N, K, dtype, la, lb, *_ = inputs.WORKLOADS[name]
    return dict(name=name, M=M, N=N, K=K, dtype=dtype, layout_a=la, layout_b=lb)


def test_rotation_keeps_the_operands_in_flight_above_twice_the_l2():
    want = {"square8192_bf16": 1, "wave2304_bf16": 4, "mlp8192x14336x4096_bf16": 2,
            "skinny64x8192x8192_f16": 2, "square512_f16": 247}
    for name, copies in want.items():
        spec = _spec(name)
        assert bench.rotation_copies(spec) == copies, name
        ab = 2.0 * (spec["M"] * spec["K"] + spec["K"] * spec["N"])
        assert copies * ab > 2 * bench.L2_BYTES
        note = bench.l2_note(spec)
        assert ("rotated over %d copies" % copies in note) == (copies > 1)


class _FakePlan:
    def __init__(self, schedule, sk_mode, split_cluster=0):
        self._info = {"schedule": schedule, "sk_mode": sk_mode, "split_k_cluster": split_cluster}

    def info(self, key):
        return self._info[key]


def test_auto_files_its_traffic_under_the_schedule_it_resolves_to():
    assert bench.resolved_name("persistent", _FakePlan(2, 1)) == "persistent"
    assert bench.resolved_name("auto", _FakePlan(1, 0)) == "persistent"
    assert bench.resolved_name("auto", _FakePlan(2, 0)) == "streamk"
    assert bench.resolved_name("auto", _FakePlan(2, 1)) == "streamk_all"
    assert bench.resolved_name("auto", _FakePlan(3, 0)) == "splitk"
    assert bench.resolved_name("auto", _FakePlan(3, 0, 1)) == "splitk_cluster"
    assert bench.resolved_name("auto", _FakePlan(0, 0)) == "dp"


def test_traffic_is_read_only_for_the_current_kernel_sources(tmp_path, monkeypatch):
    sha = bench.kernel_source_hash()
    (tmp_path / "profiles").mkdir()
    f = tmp_path / "profiles" / "gemm_kernel_streamk_square8192_bf16.md"
    f.write_text("summary\n\ntraffic_bytes_per_launch: 1234567\nkernel_source_sha: %s\n"
                 % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: sha)
    assert bench.profiled_traffic("square8192_bf16", "streamk") == 1234567.0
    assert bench.profiled_traffic("square8192_bf16", "persistent") is None      # no summary
    f.write_text("traffic_bytes_per_launch: 1234567\nkernel_source_sha: 0000000000000000\n")
    assert bench.profiled_traffic("square8192_bf16", "streamk") is None         # stale counters


def test_committed_summaries_carry_traffic_and_source_hash():
    import os, re
    names = [n for n in os.listdir(os.path.join(bench.ROOT, "profiles"))
             if n.startswith("gemm_kernel_")]
    assert names
    for n in names:
        text = open(os.path.join(bench.ROOT, "profiles", n)).read()
        assert re.search(r"traffic_bytes_per_launch:\s*[0-9]", text), n
        assert re.search(r"kernel_source_sha:\s*[0-9a-f]{16}", text), n
