"""GPU parity at large sizes: a tall product, a very deep K on a small output
(long Stream-K and split-K ranges, eight 32768-deep parts of cluster split-K),
and a wide N (cluster split-K in waves of 2-CTA clusters); sampled entries
against the oracle, integer-valued operands bit-exact."""
import numpy as np
import pytest

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs, tune
from tests.gpu_util import Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # M, N, K, dtype, layout A, layout B, schedules
    (16384, 2048, 4096, inputs.BF16, 0, 1, ("persistent", "streamk", "auto")),
    (256, 256, 262144, inputs.BF16, 0, 1, ("streamk", "splitk", "splitk_cluster", "auto")),
    (128, 65536, 1024, inputs.F16, 0, 0, ("dp", "streamk", "splitk_cluster", "auto")),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    oracle.build()


@pytest.mark.parametrize("M,N,K,dtype,la,lb,scheds", CASES)
def test_large(M, N, K, dtype, la, lb, scheds):
    rng = np.random.default_rng(M + N + K)
    rows = np.concatenate([rng.integers(0, M, 4000), [0, M - 1, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 4000), [N - 1, 0, N - 1]])
    ws = Workspace()
    for law in (("normal", 1.0), inputs.INT_LAW):
        A, Bm = inputs.operands(M, N, K, dtype, la, lb, law, law, seed=K % 1000 + M % 1000)
        dA, dB = to_device(A), to_device(Bm)
        C64, S = oracle.gemm_entries(A, Bm, M, N, K, dtype, la, lb, rows, cols)
        ref = oracle.round_to(C64, dtype)
        for sched in scheds:
            kind, opts = tune.SCHEDULE_VARIANTS[sched]
            p = B.Plan(M, N, K, dtype, la, lb, kind, **opts)
            got = run(p, dA, dB, M, N, ws)[rows, cols]
            p.close()
            ok, worst, nbad = oracle.check(got, dtype, C64, S, K)
            assert ok, (M, N, K, sched, nbad, worst)
            if law == inputs.INT_LAW:
                assert np.array_equal(got, ref), (M, N, K, sched)
