"""GPU parity on the five measured workloads at full size, in the launch
configuration the benchmark times (default plan options of every schedule it
times, AUTO included).

Every element of C is compared with the oracle's full product: real-valued
inputs within the acceptance bound, integer-valued inputs bit-exact.  Every
schedule must also be bitwise identical run to run.  The oracle computes
the 8192^3 product in about 10-20 s on the host cores."""
import numpy as np
import pytest

import oracle
from persistent_stream_matmul_gb300 import inputs
from persistent_stream_matmul_gb300 import _binding as B
from tests.gpu_util import Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

# the schedules bench.py times, with its option sets
SCHEDS = {"dp": ("dp", {}), "persistent": ("persistent", {}), "streamk": ("streamk", {}),
          "streamk_all": ("streamk", {"sk_mode": 1}), "splitk": ("splitk", {}),
          "splitk_cluster": ("splitk", {"split_cluster": 1}), "auto": ("auto", {})}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    oracle.build()


@pytest.mark.parametrize("integer", [False, True], ids=["real", "int"])
@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_full(name, integer):
    spec, A, Bm = inputs.workload(name, integer=integer)
    M, N, K, dtype = spec["M"], spec["N"], spec["K"], spec["dtype"]
    la, lb = spec["layout_a"], spec["layout_b"]
    dA, dB = to_device(A), to_device(Bm)
    ws = Workspace()
    # integer inputs: every partial sum is an exact integer, so the rounded
    # oracle value is the only correct answer and the bound is not needed
    C64, S, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb, with_abs=not integer)
    outs = {}
    for sched, (kind, opts) in SCHEDS.items():
        p = B.Plan(M, N, K, dtype, la, lb, kind, **opts)
        Cb = run(p, dA, dB, M, N, ws)
        if integer:
            nbad = int(np.count_nonzero(Cb != Cref))
            assert nbad == 0, (name, sched, nbad)
        else:
            ok, worst, nbad = oracle.check(Cb, dtype, C64, S, K)
            assert ok, (name, sched, nbad, worst)
        # run to run: bitwise identical
        assert np.array_equal(run(p, dA, dB, M, N, ws), Cb), (name, sched)
        outs[sched] = Cb
        p.close()
    if integer:
        for sched in SCHEDS:
            assert np.array_equal(outs["dp"], outs[sched]), sched
