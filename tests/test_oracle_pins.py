"""Pins for the CPU oracle: each check compares it with something other than
itself (a library conversion, exact rational arithmetic, integer arithmetic,
an algebraic identity), chosen so that a dropped term, a wrong sign or index,
or a transposed operand in the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from persistent_stream_matmul_gb300 import inputs

F16, BF16 = 0, 1
FMT = {F16: (11, -14, 15), BF16: (8, -126, 127)}   # significand bits, emin, emax


# ---------------------------------------------------------------------------
# textbook round-to-nearest-even on exact rationals (independent of the C code)
# ---------------------------------------------------------------------------
def rne_fraction(x: Fraction, dtype: int) -> Fraction:
    """Nearest representable value (ties to even significand), inf as None."""
    p, emin, emax = FMT[dtype]
    if x == 0:
        return Fraction(0)
    a = abs(x)
    # exponent e with 2^e <= a < 2^(e+1), floored at emin (subnormals)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    q = Fraction(2) ** (e - (p - 1))            # spacing of the grid at a
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    largest = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > largest:
        return None
    return r if x > 0 else -r


def value_of_bits(h: int, dtype: int):
    """Independent decoder used only to read the textbook result back."""
    if dtype == F16:
        return float(np.array([h], dtype=np.uint16).view(np.float16)[0])
    return float(np.array([h << 16], dtype=np.uint32).view(np.float32)[0])


# ---------------------------------------------------------------------------
# 16-bit formats
# ---------------------------------------------------------------------------
def test_decode_every_f16_pattern_matches_numpy(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_decode_every_bf16_pattern_is_top_half_of_fp32(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode(bits, BF16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def _probe_doubles(rng, dtype):
    p, emin, emax = FMT[dtype]
    # random magnitudes across the whole range, including subnormals
    exps = rng.integers(emin - p - 2, emax + 2, size=4000)
    x = rng.uniform(1.0, 2.0, size=exps.size) * np.ldexp(1.0, exps)
    x *= rng.choice([-1.0, 1.0], size=x.size)
    # exact midpoints between neighbours (ties), normal and subnormal
    vals = np.arange(0, 2 ** 15, 7, dtype=np.uint16)
    lo = np.abs(np.array([value_of_bits(int(h), dtype) for h in vals]))
    hi = np.abs(np.array([value_of_bits(int(h) + 1, dtype) for h in vals]))
    fin = np.isfinite(lo) & np.isfinite(hi)
    mids = (lo[fin] + hi[fin]) / 2          # exact in double
    largest = (2 - 2.0 ** (1 - p)) * 2.0 ** emax
    edge = [0.0, -0.0, largest, -largest, (2 - 2.0 ** -p) * 2.0 ** emax,
            np.nextafter((2 - 2.0 ** -p) * 2.0 ** emax, 0), 2.0 ** emin,
            2.0 ** (emin - p + 1), 2.0 ** (emin - p), 3 * 2.0 ** (emin - p),
            np.nextafter(2.0 ** (emin - p), 0), np.nextafter(2.0 ** (emin - p), 1)]
    return np.concatenate([x, mids, -mids, np.array(edge)])


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_round_matches_textbook_definition(oracle_mod, dtype):
    rng = np.random.default_rng(7 + dtype)
    x = _probe_doubles(rng, dtype)
    got = oracle_mod.round_to(x, dtype)
    for xi, hi in zip(x.tolist(), got.tolist()):
        ref = rne_fraction(Fraction(xi), dtype)
        v = value_of_bits(hi, dtype)
        if ref is None:
            assert np.isinf(v) and np.sign(v) == np.sign(xi), (xi, hi)
        else:
            assert Fraction(v) == ref, (xi, hi, v, float(ref))
            if xi == 0:
                assert (hi >> 15) == int(np.signbit(xi))


def test_round_f16_matches_numpy_conversion(oracle_mod):
    rng = np.random.default_rng(11)
    x = _probe_doubles(rng, F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle_mod.round_to(x, F16), ref)


def test_round_bf16_matches_torch_on_fp32_values(oracle_mod):
    # for values that are exact in fp32, torch's fp32 -> bf16 cast is one RNE
    rng = np.random.default_rng(12)
    x = _probe_doubles(rng, BF16).astype(np.float32).astype(np.float64)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    ref = ref.numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.round_to(x, BF16), ref)


def test_round_is_direct_not_through_fp32(oracle_mod):
    # 1 + 2^-8 + 2^-30 is just above a bf16 tie; going through fp32 first
    # drops the 2^-30 and lands on the tie, which rounds down to 1.0
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -11 + 2.0 ** -40])
    got_bf = oracle_mod.round_to(x[:1], BF16)[0]
    got_h = oracle_mod.round_to(x[1:], F16)[0]
    assert value_of_bits(int(got_bf), BF16) == 1.0 + 2.0 ** -7
    assert value_of_bits(int(got_h), F16) == 1.0 + 2.0 ** -10


# ---------------------------------------------------------------------------
# the product
# ---------------------------------------------------------------------------
def _exact_product(A, B, M, N, K, dtype, la, lb):
    """Brute-force i-j-k loop over exact rationals from the decoded inputs."""
    def a_at(i, k):
        return Fraction(value_of_bits(int(A[i, k] if la == 0 else A[k, i]), dtype))

    def b_at(k, j):
        return Fraction(value_of_bits(int(B[k, j] if lb == 0 else B[j, k]), dtype))

    C = [[Fraction(0)] * N for _ in range(M)]
    S = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            c = s = Fraction(0)
            for k in range(K):
                x, y = a_at(i, k), b_at(k, j)
                c += x * y
                s += abs(x) * abs(y)
            C[i][j], S[i][j] = c, s
    return C, S


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("la,lb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_brute_force_tiny_shapes(oracle_mod, dtype, la, lb):
    rng = np.random.default_rng(100 + 10 * dtype + 2 * la + lb)
    for trial in range(6):
        M, N, K = (int(v) for v in rng.integers(1, 18, size=3))
        law = ("uniform", -1.0, 1.0) if trial % 2 else ("normal", 3.0)
        A, B = inputs.operands(M, N, K, dtype, la, lb, law, law, seed=1000 + trial)
        C64, S, Cb = oracle_mod.gemm(A, B, M, N, K, dtype, la, lb)
        Cx, Sx = _exact_product(A, B, M, N, K, dtype, la, lb)
        for i in range(M):
            for j in range(N):
                # recursive double summation: error <= (K-1) u sum|ab|, u = 2^-53
                bound = (K - 1) * 2.0 ** -53 * float(Sx[i][j]) * (1 + 1e-12)
                assert abs(Fraction(C64[i, j]) - Cx[i][j]) <= Fraction(bound), (i, j)
                assert abs(S[i, j] - float(Sx[i][j])) <= bound
                ref = rne_fraction(Fraction(C64[i, j]), dtype)
                assert Fraction(value_of_bits(int(Cb[i, j]), dtype)) == ref


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("la,lb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_integer_inputs_are_exact(oracle_mod, dtype, la, lb):
    M, N, K = 37, 23, 301
    A, B = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, seed=77)
    a = oracle_mod.decode(A, dtype).astype(np.int64)
    b = oracle_mod.decode(B, dtype).astype(np.int64)
    a = a if la == 0 else a.T
    b = b if lb == 0 else b.T
    ref = a @ b                                   # int64 arithmetic
    C64, S, Cb = oracle_mod.gemm(A, B, M, N, K, dtype, la, lb)
    assert np.array_equal(C64, ref.astype(np.float64))
    assert np.array_equal(S, (np.abs(a) @ np.abs(b)).astype(np.float64))
    for v, h in zip(ref.ravel()[:400].tolist(), Cb.ravel()[:400].tolist()):
        assert Fraction(value_of_bits(h, dtype)) == rne_fraction(Fraction(v), dtype)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("la,lb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_identity_and_permutation(oracle_mod, dtype, la, lb):
    M, K = 19, 13
    one = int(inputs.to_bits(np.array([1.0]), dtype)[0])
    A, _ = inputs.operands(M, K, K, dtype, la, 0, ("uniform", -4.0, 4.0),
                           ("uniform", -1, 1), seed=5)
    a_log = A if la == 0 else A.T                 # logical M x K patterns
    # A * I = A
    eye = np.zeros((K, K), dtype=np.uint16)
    np.fill_diagonal(eye, one)
    _, _, Cb = oracle_mod.gemm(A, eye, M, K, K, dtype, la, lb)
    assert np.array_equal(Cb, a_log)
    # A * P = columns of A permuted: P[k, perm[k]] = 1 puts A[:, k] in column perm[k]
    perm = np.random.default_rng(3).permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), perm] = one
    Pst = P if lb == 0 else np.ascontiguousarray(P.T)
    _, _, Cb = oracle_mod.gemm(A, Pst, M, K, K, dtype, la, lb)
    expect = np.empty_like(a_log)
    expect[:, perm] = a_log
    assert np.array_equal(Cb, expect)
    # I * B = B with B non-square (K x N)
    N = 29
    _, B = inputs.operands(K, N, K, dtype, 0, lb, ("uniform", -1, 1),
                           ("uniform", -4.0, 4.0), seed=6)
    b_log = B if lb == 0 else B.T
    _, _, Cb = oracle_mod.gemm(eye, B, K, N, K, dtype, la, lb)
    assert np.array_equal(Cb, b_log)


def test_transposed_operand_is_caught(oracle_mod):
    # a planted mistake (reading B with the wrong layout) breaks the pin
    dtype, M, K = F16, 9, 9
    one = int(inputs.to_bits(np.array([1.0]), dtype)[0])
    A, _ = inputs.operands(M, K, K, dtype, 0, 0, ("uniform", -4, 4), ("uniform", -1, 1), 5)
    perm = np.roll(np.arange(K), 1)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), perm] = one
    _, _, good = oracle_mod.gemm(A, P, M, K, K, dtype, 0, 0)
    _, _, bad = oracle_mod.gemm(A, P, M, K, K, dtype, 0, 1)
    assert not np.array_equal(good, bad)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_associativity_invariant(oracle_mod, dtype):
    M, N, K = 48, 40, 200
    A, B = inputs.operands(M, N, K, dtype, 0, 1, ("normal", 1.0), ("normal", 1.0), seed=9)
    C64, S, _ = oracle_mod.gemm(A, B, M, N, K, dtype, 0, 1)
    a = oracle_mod.decode(A, dtype)
    b = oracle_mod.decode(B, dtype).T
    x = np.random.default_rng(1).normal(size=N)
    lhs = C64 @ x
    rhs = a @ (b @ x)
    scale = np.abs(a) @ (np.abs(b) @ np.abs(x))
    assert np.all(np.abs(lhs - rhs) <= 2 * K * N * 2.0 ** -52 * scale)
    # a dropped k term (last column of A zeroed) must break it
    a2 = a.copy()
    a2[:, -1] = 0
    assert not np.all(np.abs(lhs - a2 @ (b @ x)) <= 2 * K * N * 2.0 ** -52 * scale)


def test_entries_agree_with_full_product(oracle_mod):
    M, N, K, dtype = 70, 90, 333, BF16
    A, B = inputs.operands(M, N, K, dtype, 0, 1, ("normal", 1.0), ("normal", 1.0), seed=4)
    C64, S, _ = oracle_mod.gemm(A, B, M, N, K, dtype, 0, 1)
    rng = np.random.default_rng(0)
    r = rng.integers(0, M, 500)
    c = rng.integers(0, N, 500)
    e64, es = oracle_mod.gemm_entries(A, B, M, N, K, dtype, 0, 1, r, c)
    assert np.array_equal(e64, C64[r, c])
    assert np.array_equal(es, S[r, c])


def test_empty_and_zero_k(oracle_mod):
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((0, 4), dtype=np.uint16)
    C64, S, Cb = oracle_mod.gemm(A, B, 3, 4, 0, F16)
    assert not C64.any() and not S.any() and not Cb.any()
    C64, S, Cb = oracle_mod.gemm(np.zeros((0, 5), np.uint16), np.zeros((5, 2), np.uint16),
                                 0, 2, 5, F16)
    assert C64.shape == (0, 2)


# ---------------------------------------------------------------------------
# the acceptance check
# ---------------------------------------------------------------------------
def test_check_accepts_just_inside_and_rejects_just_outside(oracle_mod):
    K = 1000
    C64 = np.array([1.0, -3.0, 0.0, 2.0 ** -20])
    S = np.array([50.0, 10.0, 0.0, 1.0])
    bound = oracle_mod.tolerance_bound(C64, S, K)
    assert np.allclose(bound, 2.0 ** -8 * np.abs(C64) + K * 2.0 ** -22 * S)
    inside = oracle_mod.round_to(C64 + 0.5 * bound, BF16)
    ok, worst, nbad = oracle_mod.check(inside, BF16, C64, S, K)
    assert ok and worst <= 1.0 and nbad == 0
    outside = oracle_mod.round_to(C64[:2] + 3 * bound[:2], BF16)
    ok, worst, nbad = oracle_mod.check(outside, BF16, C64[:2], S[:2], K)
    assert not ok and nbad == 2
    # an exact zero with an empty sum must be exactly zero
    ok, _, _ = oracle_mod.check(oracle_mod.round_to(np.array([1e-30]), F16),
                                F16, np.array([0.0]), np.array([0.0]), K)
    assert ok   # 1e-30 rounds to 0 in fp16
    ok, _, _ = oracle_mod.check(oracle_mod.round_to(np.array([1e-3]), F16),
                                F16, np.array([0.0]), np.array([0.0]), K)
    assert not ok
