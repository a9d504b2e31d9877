"""The seeded operand generator shared by the GPU tests, the benchmark and the
oracle checks."""
import numpy as np

from persistent_stream_matmul_gb300 import inputs


def test_splitmix64_published_outputs():
    # the first outputs of splitmix64 started from state 0
    got = [int(v) for v in inputs.splitmix64(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_offsets_are_consistent():
    a = inputs.splitmix64(1234, 10)
    b = inputs.splitmix64(1234, 4, offset=6)
    assert np.array_equal(a[6:], b)


def test_laws():
    u = inputs.draw(("uniform", -1.0, 1.0), 7, 200000)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    n = inputs.draw(("normal", 2.0), 7, 200000)
    assert abs(n.mean()) < 0.02 and abs(n.std() - 2.0) < 0.02
    i = inputs.draw(("int", -2, 2), 7, 200000)
    vals, counts = np.unique(i, return_counts=True)
    assert vals.tolist() == [-2, -1, 0, 1, 2] and counts.min() > 39000


def test_bf16_rounding_matches_fp32_route_when_exact():
    x = np.random.default_rng(0).normal(size=10000).astype(np.float32).astype(np.float64)
    got = inputs.to_bits(x, inputs.BF16)
    # for fp32-exact values, rounding the fp32 bit pattern is the same RNE
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    ref = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(got, ref)


def test_storage_shapes_and_determinism():
    spec, A, B = inputs.workload("square512_f16")
    assert A.shape == (512, 512) and B.shape == (512, 512) and A.dtype == np.uint16
    _, A2, B2 = inputs.workload("square512_f16")
    assert np.array_equal(A, A2) and np.array_equal(B, B2)
    _, Ai, _ = inputs.workload("square512_f16", integer=True)
    v = Ai.view(np.float16).astype(np.float64)
    assert set(np.unique(v).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}
    A, B = inputs.operands(5, 7, 3, inputs.BF16, inputs.COL_MAJOR, inputs.COL_MAJOR,
                           ("normal", 1.0), ("normal", 1.0), 1)
    assert A.shape == (3, 5) and B.shape == (7, 3)


def test_chunked_draws_equal_one_draw():
    # the generator pool cuts operands into chunks; the bytes must not change
    for law in (("uniform", -1.0, 1.0), ("normal", 0.5), ("int", -2, 2)):
        for dtype in (inputs.F16, inputs.BF16):
            whole = inputs.to_bits(inputs.draw(law, 99, 1000), dtype).reshape(40, 25)
            for chunk in (1, 7, 64, 999, 1000, 5000):
                got = inputs.matrix(40, 25, inputs.ROW_MAJOR, dtype, law, 99 >> 8, 99 & 255,
                                    chunk=chunk)
                assert np.array_equal(got, whole), (law, dtype, chunk)


def test_operand_bytes_are_stable():
    # digests of the operands as the generator first produced them: the
    # workloads' bytes must not change when the generator is reorganised
    import hashlib
    want = {(("uniform", -1.0, 1.0), 0): "6fd08b0bafdb0e3e", (("uniform", -1.0, 1.0), 1): "785c5cf6eca36cfb",
            (("normal", 0.5), 0): "0dcdf3c465b4364f", (("normal", 0.5), 1): "fcc231cb818faf82",
            (("int", -2, 2), 0): "8e0590bd0c8ac4ec", (("int", -2, 2), 1): "fb21f0fc867db2b1"}
    for (law, dtype), digest in want.items():
        for chunk in (inputs.CHUNK, 4096):
            b = inputs.matrix(300, 70, inputs.ROW_MAJOR, dtype, law, 0x5EED0001, 1, chunk=chunk)
            assert hashlib.sha256(b.tobytes()).hexdigest()[:16] == digest, (law, dtype, chunk)
