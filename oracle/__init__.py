"""Oracle for the double-double GEMM: plain, slow, obviously correct CPU code.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may load it.  It shares no code, header, table or
constant generator with the CUDA library in ``extended_precision_gemm_gb300``;
the two meet only in the seeded input generator (``workloads``).

Two parts:

* ``exact_dd_gemm`` (C, ``exact_ddgemm.c``): the plain definition of the
  product.  Every product of the four double pairs is formed exactly and added
  into a wide fixed-point superaccumulator, which is rounded once to the
  nearest double double ("Multiple Double Arithmetic on NVIDIA Tensor Cores",
  Definition 1.1 and the last step of the Section 2 algorithm).
* ``oracle.slices``: the method's own steps in the page's order (shared
  exponents, 13-bit quarters, slice-pair products grouped by index sum,
  double-double recombination), written from the page's description.  The GPU
  path's intermediate results are compared with these bit for bit.

Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``): exact rational brute
force on tiny inputs, identity and permutation matrices, closed forms,
transposition / scaling / negation / k-order invariants, the worked quartering
example of Section 2, and the bound of eq. (5).
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import threading

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "exact_ddgemm.c"
_BUILD_DIR = _HERE / "_build"
_LIB_PATH = _BUILD_DIR / "liboracle.so"
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> pathlib.Path:
    """Compile exact_ddgemm.c with gcc + OpenMP into oracle/_build/liboracle.so."""
    _BUILD_DIR.mkdir(exist_ok=True)
    if not force and _LIB_PATH.exists() and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    tmp = _BUILD_DIR / f"liboracle.{os.getpid()}.so"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build()))
            f = lib.oracle_dd_gemm_block
            f.restype = ctypes.c_int
            i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            f.argtypes = [i64, i64, i64, dp, dp, i64, dp, dp, i64,
                          i64, ip, i64, ip, dp, dp, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            g = lib.oracle_md_gemm_block
            g.restype = ctypes.c_int
            g.argtypes = [ctypes.c_int, i64, i64, i64, dp, i64, dp, i64, i64, ip, i64, ip, dp, ctypes.c_int]
            _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP loop uses by default (all host cores)."""
    return int(_load().oracle_max_threads())


def _f64(x):
    a = np.ascontiguousarray(x, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("matrices must be 2-D")
    return a


def exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=None, cols=None, threads: int = 0):
    """Exact C = (A_hi + A_lo) @ (B_hi + B_lo), rounded once to the nearest dd.

    Returns (C_hi, C_lo) for the rows ``rows`` and columns ``cols`` of C
    (all of them by default), as float64 arrays of shape (len(rows), len(cols)).
    """
    A_hi, A_lo, B_hi, B_lo = map(_f64, (A_hi, A_lo, B_hi, B_lo))
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if A_lo.shape != (M, K) or B_lo.shape != (K2, N) or K2 != K:
        raise ValueError("shape mismatch")
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    out_hi = np.zeros((rows.size, cols.size), dtype=np.float64)
    out_lo = np.zeros((rows.size, cols.size), dtype=np.float64)
    rc = _load().oracle_dd_gemm_block(
        M, N, K, A_hi.ctypes.data, A_lo.ctypes.data, K, B_hi.ctypes.data, B_lo.ctypes.data, N,
        rows.size, rows.ctypes.data, cols.size, cols.ctypes.data,
        out_hi.ctypes.data, out_lo.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError({1: "bad argument", 2: "non-finite input", 3: "out of host memory"}.get(rc, rc))
    return out_hi, out_lo


def exact_md_gemm(A_parts, B_parts, rows=None, cols=None, threads: int = 0):
    """Exact product of multiple-double matrices (A = sum of the planes in
    A_parts, B likewise), rounded once into len(A_parts) non-overlapping
    doubles: x_0 = RN(X), x_1 = RN(X - x_0), ...  Returns the list of part
    planes for the chosen rows and columns."""
    A_parts = [_f64(a) for a in A_parts]
    B_parts = [_f64(b) for b in B_parts]
    np_ = len(A_parts)
    if len(B_parts) != np_:
        raise ValueError("A and B need the same number of parts")
    M, K = A_parts[0].shape
    K2, N = B_parts[0].shape
    if K2 != K or any(a.shape != (M, K) for a in A_parts) or any(b.shape != (K, N) for b in B_parts):
        raise ValueError("shape mismatch")
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    outs = [np.zeros((rows.size, cols.size)) for _ in range(np_)]
    PtrArr = ctypes.c_void_p * np_
    a_ptrs = PtrArr(*[a.ctypes.data for a in A_parts])
    b_ptrs = PtrArr(*[b.ctypes.data for b in B_parts])
    o_ptrs = PtrArr(*[o.ctypes.data for o in outs])
    rc = _load().oracle_md_gemm_block(np_, M, N, K, ctypes.cast(a_ptrs, ctypes.c_void_p), K,
                                      ctypes.cast(b_ptrs, ctypes.c_void_p), N,
                                      rows.size, rows.ctypes.data, cols.size, cols.ctypes.data,
                                      ctypes.cast(o_ptrs, ctypes.c_void_p), int(threads))
    if rc != 0:
        raise ValueError({1: "bad argument", 2: "non-finite input", 3: "out of host memory"}.get(rc, rc))
    return outs
