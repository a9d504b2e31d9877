"""CPU oracle for C = A*B with fp16/bf16 inputs, and for the Stream-K schedule.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check
(``__graft_entry__.smoke``) and the benchmark's CPU-baseline leg may import
this package.  The GPU library never imports, links or calls it, and it never
imports the GPU library.

Two parts:

* ``oracle_gemm.c`` (loaded here with ctypes): the plain product in double
  precision, one direct rounding to the 16-bit output type, and the sum of
  |a||b| used by the acceptance bound.  See the file header for the citation.
* ``streamk_schedule``: the work decomposition of the Triton Stream-K kernel
  in the issue "Stream-k matmul implementation very slow" (final version),
  restated in plain Python.

Parity is pinned for every function here by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gemm.so")

F16, BF16 = 0, 1
ROW_MAJOR, COL_MAJOR = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` into ``liboracle_gemm.so`` (gcc + OpenMP).

    No fast-math and no FMA contraction: the sum is plain IEEE double in
    ascending k.
    """
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = [
            "gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
            "-fno-fast-math", "-ffp-contract=off", "-fno-strict-aliasing",
            _SRC, "-o", tmp, "-lm",
        ]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_decode.argtypes = [i32, vp, i64, vp]
        lib.oracle_round.argtypes = [i32, vp, i64, vp]
        lib.oracle_gemm.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.oracle_gemm_entries.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp,
                                            i64, vp, vp, vp, vp]
        lib.oracle_num_threads.argtypes = []
        for f in (lib.oracle_decode, lib.oracle_round, lib.oracle_gemm,
                  lib.oracle_gemm_entries, lib.oracle_num_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle uses (``OMP_NUM_THREADS`` or all cores)."""
    return int(_load().oracle_num_threads())


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact value of each 16-bit pattern, as float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().oracle_decode(int(dtype), _ptr(bits), bits.size, _ptr(out))
    if rc:
        raise ValueError("oracle_decode: bad dtype %r" % dtype)
    return out


def round_to(x: np.ndarray, dtype: int) -> np.ndarray:
    """float64 -> 16-bit patterns, one rounding, to nearest with ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    rc = _load().oracle_round(int(dtype), _ptr(x), x.size, _ptr(out))
    if rc:
        raise ValueError("oracle_round: bad dtype %r" % dtype)
    return out


def gemm(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, dtype: int,
         layout_a: int = ROW_MAJOR, layout_b: int = ROW_MAJOR, with_abs: bool = True):
    """Full product.  ``A``/``B`` are uint16 patterns in the stated layouts.

    Returns ``(C64, S, Cbits)``: the double-precision sum (M x N), the sum of
    |a||b| (or None) and the output rounded once to ``dtype`` (uint16 M x N).
    """
    A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.uint16).reshape(-1)
    if A.size != M * K or B.size != K * N:
        raise ValueError("operand sizes do not match M, N, K")
    C64 = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    Cb = np.empty((M, N), dtype=np.uint16)
    rc = _load().oracle_gemm(M, N, K, int(dtype), int(layout_a), int(layout_b),
                             _ptr(A), _ptr(B), _ptr(C64), _ptr(S), _ptr(Cb))
    if rc:
        raise RuntimeError("oracle_gemm failed with code %d" % rc)
    return C64, S, Cb


def gemm_entries(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, dtype: int,
                 layout_a: int, layout_b: int, rows, cols):
    """Selected entries (rows[e], cols[e]) of the product: ``(C64, S)``."""
    A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.uint16).reshape(-1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in shape")
    C64 = np.empty(rows.shape, dtype=np.float64)
    S = np.empty(rows.shape, dtype=np.float64)
    rc = _load().oracle_gemm_entries(M, N, K, int(dtype), int(layout_a), int(layout_b),
                                     _ptr(A), _ptr(B), rows.size, _ptr(rows), _ptr(cols),
                                     _ptr(C64), _ptr(S))
    if rc:
        raise RuntimeError("oracle_gemm_entries failed with code %d" % rc)
    return C64, S


def tolerance_bound(C64: np.ndarray, S: np.ndarray, K: int) -> np.ndarray:
    """Elementwise acceptance bound 2^-8*|C_ref| + K*2^-22*sum_k|a_ik||b_kj|.

    The bound is stated for the fp32-accumulated, once-rounded result; the
    first term covers one bf16 rounding (unit roundoff 2^-8), the second four
    times the textbook bound K*2^-24*sum|a||b| of a length-K fp32 sum.
    """
    return np.ldexp(np.abs(C64), -8) + float(K) * np.ldexp(S, -22)


def check(C_bits: np.ndarray, dtype: int, C64: np.ndarray, S: np.ndarray, K: int):
    """Compare a 16-bit result against the oracle under the acceptance bound.

    Returns ``(ok, worst_ratio, n_bad)`` where worst_ratio is
    max |C - C64| / bound (0/0 counts as 0, x/0 as inf).
    """
    got = decode(np.asarray(C_bits, dtype=np.uint16), dtype)
    err = np.abs(got - C64)
    bound = tolerance_bound(C64, S, K)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(err == 0, 0.0, err / bound)
    bad = ~(err <= bound)
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return (not bool(bad.any())), worst, int(bad.sum())
