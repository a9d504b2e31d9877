"""Seeded synthetic operands for C = A*B (fp16 / bf16).

This module is the one piece shared by the GPU path's tests and benchmark and
by the CPU oracle's checks: both are fed the bytes it makes.  It holds none of
the product's arithmetic, only random numbers and their rounding to the input
type.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", 2014) run as a counter-based stream: output i of stream
``key`` is mix64(key + (i + 1) * 0x9E3779B97F4A7C15), where mix64 is the
published finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
multiply 0x94D049BB133111EB, xor-shift 31).  The top 53 bits give a uniform
double in [0, 1).  Normals come from the Box-Muller transform.  Values are
drawn in storage order, then rounded once from double to the input type,
to nearest with ties to even.

Workload recipes (matrix shapes, types, layouts, value laws) are the five
workloads the library is measured on; see ``WORKLOADS``.
"""
from __future__ import annotations

import os

import numpy as np

F16, BF16 = 0, 1
ROW_MAJOR, COL_MAJOR = 0, 1

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# name: (M, N, K, dtype, layout A, layout B, law A, law B, seed)
# law: ("uniform", lo, hi) | ("normal", sigma) | ("int", lo, hi)
WORKLOADS = {
    "square512_f16": (512, 512, 512, F16, ROW_MAJOR, ROW_MAJOR,
                      ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), 0x5EED0001),
    "square8192_bf16": (8192, 8192, 8192, BF16, ROW_MAJOR, COL_MAJOR,
                        ("normal", 8192 ** -0.5), ("normal", 8192 ** -0.5), 0x5EED0002),
    "wave2304_bf16": (2304, 2304, 8192, BF16, ROW_MAJOR, COL_MAJOR,
                      ("normal", 8192 ** -0.5), ("normal", 8192 ** -0.5), 0x5EED0003),
    "mlp8192x14336x4096_bf16": (8192, 14336, 4096, BF16, ROW_MAJOR, COL_MAJOR,
                                ("normal", 1.0), ("normal", 0.02), 0x5EED0004),
    "skinny64x8192x8192_f16": (64, 8192, 8192, F16, ROW_MAJOR, ROW_MAJOR,
                               ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), 0x5EED0005),
}
INT_LAW = ("int", -2, 2)
INT_SEED_OFFSET = 100


def splitmix64(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the counter-based splitmix64 stream."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key & 0xFFFFFFFFFFFFFFFF) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Doubles in [0, 1): top 53 bits of the stream times 2^-53."""
    return (splitmix64(key, n, offset) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def draw(law, key: int, n: int) -> np.ndarray:
    """n doubles from a value law: ``uniform`` (lo, hi) scales the uniform
    doubles; ``normal`` (sigma) takes pairs of them through Box-Muller,
    sqrt(-2 ln(1 - u1)) cos(2 pi u2); ``int`` (lo, hi) maps the top 53 bits
    of each output to lo .. hi by a multiply-shift."""
    return draw_range(law, key, 0, n)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round doubles to 16-bit patterns (to nearest, ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == F16:
        with np.errstate(over="ignore"):
            return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        a = np.abs(x)
        if np.any((a != 0) & (a < 2.0 ** -126)) or np.any(a >= 2.0 ** 127):
            raise ValueError("bf16 input generator: value outside the normal range")
        b = x.view(np.uint64)
        # keep 7 stored fraction bits of the 52: drop 45, round to nearest even
        lsb = (b >> np.uint64(45)) & np.uint64(1)
        with np.errstate(over="ignore"):
            b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
        f = b.view(np.float64).astype(np.float32)   # exact: 8 significant bits
        return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError("unknown dtype %r" % dtype)


def draw_range(law, key: int, start: int, n: int) -> np.ndarray:
    """Values start .. start+n-1 of ``draw(law, key, total)`` for any total
    above start+n: every law reads the counter-based stream at fixed
    positions (value i of the normal law uses outputs 2i and 2i+1)."""
    kind = law[0]
    if kind == "uniform":
        lo, hi = law[1], law[2]
        return lo + (hi - lo) * uniform01(key, n, start)
    if kind == "normal":
        sigma = law[1]
        u = uniform01(key, 2 * n, 2 * start)
        u1 = 1.0 - u[0::2]
        u2 = u[1::2]
        return sigma * (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2))
    if kind == "int":
        lo, hi = law[1], law[2]
        width = np.uint64(hi - lo + 1)
        top = splitmix64(key, n, start) >> np.uint64(11)
        idx = (top * width) >> np.uint64(53)
        return idx.astype(np.float64) + lo
    raise ValueError("unknown law %r" % (law,))


CHUNK = 1 << 22   # values per generator task


def matrix(rows: int, cols: int, layout: int, dtype: int, law, seed: int, matrix_id: int,
           chunk: int = CHUNK):
    """A rows x cols operand as uint16 patterns in its storage shape.

    Row-major storage has shape (rows, cols); column-major storage has shape
    (cols, rows), i.e. element (r, c) is ``out[c, r]``.  Large operands are
    drawn in chunks on a thread pool (numpy releases the interpreter lock);
    the stream is counter-based, so the bytes do not depend on the chunking.
    """
    key = (seed << 8) | matrix_id
    n = rows * cols
    bits = np.empty(n, dtype=np.uint16)

    def fill(start):
        m = min(chunk, n - start)
        bits[start:start + m] = to_bits(draw_range(law, key, start, m), dtype)

    starts = range(0, n, chunk)
    if len(starts) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    elif n:
        fill(0)
    shape = (rows, cols) if layout == ROW_MAJOR else (cols, rows)
    return bits.reshape(shape)


def operands(M: int, N: int, K: int, dtype: int, layout_a: int, layout_b: int,
             law_a, law_b, seed: int):
    """(A, B) for an M x N x K product; A is M x K, B is K x N."""
    A = matrix(M, K, layout_a, dtype, law_a, seed, 1)
    B = matrix(K, N, layout_b, dtype, law_b, seed, 2)
    return A, B


def workload(name: str, integer: bool = False):
    """(spec, A, B) for a named workload; ``integer`` draws U{-2..2} instead."""
    M, N, K, dtype, la, lb, law_a, law_b, seed = WORKLOADS[name]
    if integer:
        law_a = law_b = INT_LAW
        seed += INT_SEED_OFFSET
    A, B = operands(M, N, K, dtype, la, lb, law_a, law_b, seed)
    spec = dict(name=name, M=M, N=N, K=K, dtype=dtype, layout_a=la, layout_b=lb)
    return spec, A, B
