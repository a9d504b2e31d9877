"""GPU parity over shapes drawn like the issue's log-sampled benchmark
(multiples of 256 spaced in log2 from 256 to 8192, seed 123): every schedule
and GEMM_SCHED_AUTO against the oracle on sampled entries, and bit-exact on
integer-valued operands."""
import numpy as np
import pytest

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs, tune
from tests.gpu_util import Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

VARIANTS = tune.SCHEDULE_VARIANTS
SHAPES = tune.sample_shapes(8, seed=123, max_macs=2.0 ** 33)


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    oracle.build()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_sampled_shape(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    rows = np.concatenate([rng.integers(0, M, 3000), [M - 1, 0]])
    cols = np.concatenate([rng.integers(0, N, 3000), [N - 1, N - 1]])
    ws = Workspace()
    for dtype, la, lb, law in ((inputs.BF16, 0, 1, ("normal", 1.0)),
                               (inputs.F16, 0, 0, inputs.INT_LAW)):
        A, Bm = inputs.operands(M, N, K, dtype, la, lb, law, law, seed=M ^ N ^ K)
        dA, dB = to_device(A), to_device(Bm)
        C64, S = oracle.gemm_entries(A, Bm, M, N, K, dtype, la, lb, rows, cols)
        ref = oracle.round_to(C64, dtype)
        for name, (sched, opt) in VARIANTS.items():
            p = B.Plan(M, N, K, dtype, la, lb, sched, **opt)
            got = run(p, dA, dB, M, N, ws)[rows, cols]
            p.close()
            ok, worst, nbad = oracle.check(got, dtype, C64, S, K)
            assert ok, (M, N, K, name, nbad, worst)
            if law == inputs.INT_LAW:
                assert np.array_equal(got, ref), (M, N, K, name)


def test_vs_cublas_record():
    """The comparison against torch.matmul runs and reports consistent figures
    (small product, short bursts: the record's form, not its numbers)."""
    r = tune.vs_cublas(1024, 1024, 1024, rounds=2, burst_ms=5.0)
    assert r["library_us"] > 0 and r["cublas_us"] > 0
    assert abs(r["library_tflops"] - 2.0 * 1024 ** 3 / r["library_us"] / 1e6) < 1e-6
    assert 200.0 < r["library_sm_mhz"] < 3000.0
    assert abs(r["library_kcycles"] - r["library_us"] * r["library_sm_mhz"] / 1e3) < 1e-6
    assert 0.05 < r["library_over_cublas"] < 20.0
