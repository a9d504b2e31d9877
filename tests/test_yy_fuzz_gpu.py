"""Randomized parity: random shapes, types, layouts, schedules and plan options
(tile width, clusters, pair MMA, Stream-K mode and grid, split count, cluster
split-K, raster, host-buffer pipeline), integer-valued inputs, every result bit-exact against the
CPU oracle and identical on a second run.  A fixed seed keeps it reproducible.
A sweep of this kind found a split-K host-pipeline case that the fixed tests had
missed."""
import random

import numpy as np
import pytest
import torch

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs
from tests.gpu_util import Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

CASES = 200


def _random_case(rng: random.Random):
    la, lb = rng.randint(0, 1), rng.randint(0, 1)
    M = rng.choice([1, 7, 40, 64, 65, 100, 128, 129, 200, 256, 300, 513, 640, 700, 1000, 1536])
    if la == 1:
        M = max(8, M // 8 * 8)
    N = 8 * (rng.randint(1, 150) if rng.random() < 0.8 else rng.randint(150, 400))
    K = 8 * (rng.randint(1, 400) if rng.random() < 0.8 else rng.randint(400, 1200))
    dtype = rng.choice([inputs.F16, inputs.BF16])
    sched = rng.choice(["dp", "persistent", "streamk", "splitk", "auto"])
    opt = {}
    if rng.random() < 0.7:
        opt["tile_n"] = rng.choice([64, 128, 256])
    if rng.random() < 0.5 and opt.get("tile_n", 128) != 64:
        opt["cluster_m"] = rng.choice([1, 2])
        if opt["cluster_m"] == 2:
            opt["pair_mma"] = rng.choice([0, 1])
    if sched == "streamk":
        opt["sk_mode"] = rng.choice([0, 1])
        opt["two_tiles"] = rng.choice([0, 1])
        if rng.random() < 0.4:
            opt["grid"] = rng.randint(1, 152)
    if sched == "splitk" and rng.random() < 0.5:
        opt["split_k"] = rng.randint(0, 9)
    if sched == "splitk" and rng.random() < 0.4:
        # parts reduced inside a cluster: 1-CTA tiles of 128 or 256 columns
        opt["split_cluster"] = 1
        opt["split_k"] = rng.choice([0, 2, 4, 8])
        opt.pop("cluster_m", None)
        opt.pop("pair_mma", None)
        if opt.get("tile_n") == 64:
            opt["tile_n"] = 128
    if rng.random() < 0.2:
        opt["raster"] = 1
    if rng.random() < 0.2 and sched != "dp":
        opt["group_m"] = rng.choice([0, 1, 3, 8, 16])
    host = rng.random() < 0.15
    if host:
        opt["host_chunks"] = rng.choice([0, 2, 3, 5])
    return M, N, K, dtype, la, lb, sched, opt, host


def test_random_plans_are_bit_exact_on_integers():
    ensure_built()
    oracle.build()
    rng = random.Random(20261202)
    ws = Workspace()
    stream = torch.cuda.current_stream()
    ran = 0
    for case in range(CASES):
        M, N, K, dtype, la, lb, sched, opt, host = _random_case(rng)
        A, Bm = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 3000 + case)
        _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
        try:
            p = B.Plan(M, N, K, dtype, la, lb, sched, **opt)
        except B.GemmError:
            continue                      # a combination refused at plan time
        what = (case, M, N, K, dtype, la, lb, sched, opt, host)
        if host:
            hA = torch.from_numpy(A.view(np.int16).ravel().copy()).pin_memory()
            hB = torch.from_numpy(Bm.view(np.int16).ravel().copy()).pin_memory()
            dA, dB = hA.cuda(), hB.cuda()
            dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
            for _ in range(2):
                hC = torch.full((M * N,), 0x7E5A, dtype=torch.int16).pin_memory()
                p.run_host(hA, hB, hC, dA, dB, dC, ws.get(p.workspace_size), stream)
                assert p.last_status(stream) == B.GEMM_OK, what
                assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref), what
        else:
            dA, dB = to_device(A), to_device(Bm)
            got = run(p, dA, dB, M, N, ws)
            assert np.array_equal(got, Cref), what
            assert np.array_equal(run(p, dA, dB, M, N, ws), got), what
        p.close()
        ran += 1
    assert ran >= CASES * 0.9
