"""Seeded synthetic double-double matrices for the dd GEMM workloads.

This module only draws random numbers and packs them into (hi, lo) pairs; it
holds none of the product's arithmetic.  Both the CUDA path's tests/bench and
the oracle's tests take their inputs from here.

Every matrix is a double-double pair (hi, lo) of float64 arrays with
|lo| <= ulp(hi)/2 (normalised by an error-free two-sum of hi and the drawn lo).

Draw order, per generator ``numpy.random.default_rng(seed)``: all draws for A
(the hi base values, then the per-element exponents or per-row scales where the
distribution has them, then the lo factors), then the same for B.

Workloads (double-double GEMM, C = A*B):

  0  M=N=K=64,      hi ~ U[-1,1],                       lo factor U[-1,1], seed 0
  1  M=N=K=1024,    as 0,                                                 seed 1
  2  M=N=K=4096,    hi = U[-1,1]*2^e, e ~ U{-20..20} per element, lo factor U[-1,1], seed 2
  3  M=N=256, K=65536, hi ~ N(0,1),                     lo factor N(0,1),  seed 3
  4  M=N=K=8192,    hi ~ N(0,1), A rows * 2^r, B cols * 2^c, r,c ~ U{-30..30},
                    lo factor N(0,1),                                     seed 4

lo = fp64(hi * 2^-53 * factor), then (hi, lo) <- two_sum(hi, lo).
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_dd", "make_workload", "two_sum_np", "make_md"]


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    M: int
    N: int
    K: int
    dist: str
    seed: int

    @property
    def dd_flops(self) -> float:
        """2*M*N*K: the double-double flop count the throughput metric uses."""
        return 2.0 * self.M * self.N * self.K


WORKLOADS = {
    0: Workload(0, "dd_gemm_64x64x64_uniform", 64, 64, 64, "uniform", 0),
    1: Workload(1, "dd_gemm_1024x1024x1024_uniform", 1024, 1024, 1024, "uniform", 1),
    2: Workload(2, "dd_gemm_4096x4096x4096_wide_range", 4096, 4096, 4096, "uniform_exp20", 2),
    3: Workload(3, "dd_gemm_256x256x65536_normal", 256, 256, 65536, "normal", 3),
    4: Workload(4, "dd_gemm_8192x8192x8192_scaled_normal", 8192, 8192, 8192, "normal_rowcol30", 4),
}

DISTS = ("uniform", "uniform_exp20", "normal", "normal_rowcol30")


def two_sum_np(a: np.ndarray, b: np.ndarray):
    """Error-free sum of float64 arrays (Knuth): a + b = s + e exactly."""
    s = a + b
    bb = s - a
    e = (a - (s - bb)) + (b - bb)
    return s, e


def _draw_matrix(rng: np.random.Generator, rows: int, cols: int, dist: str, scale_axis: int):
    shape = (rows, cols)
    if dist in ("uniform", "uniform_exp20"):
        hi = rng.uniform(-1.0, 1.0, shape)
        if dist == "uniform_exp20":
            ex = rng.integers(-20, 21, shape)
            hi = np.ldexp(hi, ex)
        factor = rng.uniform(-1.0, 1.0, shape)
    elif dist in ("normal", "normal_rowcol30"):
        hi = rng.standard_normal(shape)
        if dist == "normal_rowcol30":
            if scale_axis == 0:
                r = rng.integers(-30, 31, rows)
                hi = np.ldexp(hi, r[:, None])
            else:
                c = rng.integers(-30, 31, cols)
                hi = np.ldexp(hi, c[None, :])
        factor = rng.standard_normal(shape)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    lo = hi * (2.0 ** -53) * factor
    hi, lo = two_sum_np(hi, lo)
    return np.ascontiguousarray(hi), np.ascontiguousarray(lo)


def make_dd(M: int, N: int, K: int, dist: str, seed: int):
    """A (MxK) and B (KxN) double-double operands: (A_hi, A_lo, B_hi, B_lo)."""
    rng = np.random.default_rng(seed)
    A_hi, A_lo = _draw_matrix(rng, M, K, dist, scale_axis=0)
    B_hi, B_lo = _draw_matrix(rng, K, N, dist, scale_axis=1)
    return A_hi, A_lo, B_hi, B_lo


def make_workload(index: int):
    w = WORKLOADS[index]
    return make_dd(w.M, w.N, w.K, w.dist, w.seed)


def _draw_md(rng, rows, cols, dist, scale_axis, parts):
    """A multiple double with `parts` planes: x_0 as the high word of the
    distribution, then x_{p+1} = ulp(x_p)/2 * U[-1,1], which keeps every part
    below half an ulp of the previous one (non-overlapping, normalised)."""
    shape = (rows, cols)
    if dist in ("uniform", "uniform_exp20"):
        x0 = rng.uniform(-1.0, 1.0, shape)
        if dist == "uniform_exp20":
            x0 = np.ldexp(x0, rng.integers(-20, 21, shape))
    elif dist in ("normal", "normal_rowcol30"):
        x0 = rng.standard_normal(shape)
        if dist == "normal_rowcol30":
            if scale_axis == 0:
                x0 = np.ldexp(x0, rng.integers(-30, 31, rows)[:, None])
            else:
                x0 = np.ldexp(x0, rng.integers(-30, 31, cols)[None, :])
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    out = [np.ascontiguousarray(x0)]
    for _ in range(parts - 1):
        half_ulp = np.spacing(np.abs(out[-1])) * 0.5
        nxt = np.where(out[-1] == 0, 0.0, half_ulp * rng.uniform(-1.0, 1.0, shape))
        out.append(np.ascontiguousarray(nxt))
    return out


def make_md(M: int, N: int, K: int, dist: str, seed: int, parts: int = 4):
    """A (M x K) and B (K x N) multiple-double operands as lists of `parts`
    planes each (same draw order as make_dd: A's draws, then B's)."""
    rng = np.random.default_rng(seed)
    A = _draw_md(rng, M, K, dist, 0, parts)
    B = _draw_md(rng, K, N, dist, 1, parts)
    return A, B
