"""Seeded random cases through the C ABI: shapes around the tile sizes
(1, 31..33, 63..65, 127..129, 255..257), operands that are column or row
windows of larger matrices (leading dimensions above the width, base pointers
off the 16-byte grid), every distribution of the workloads, and every product
of the double-double paths -- dd_gemm, dd_gemm_ex with each fusion choice and
k-split, dd_gemm_tc -- each compared bit for bit with the oracle's model of
its method."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import workloads
from oracle import slices, slices_bf16

pytestmark = pytest.mark.gpu

EDGES = [1, 2, 7, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]
DISTS = ["uniform", "uniform_exp20", "normal", "normal_rowcol30"]


def _case(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.choice(EDGES))
    N = int(rng.choice(EDGES))
    K = int(rng.choice(EDGES + [300, 513]))
    if M * N * K > 3_000_000:      # keep the CPU model within seconds
        K = max(1, 3_000_000 // (M * N))
    return rng, M, N, K, str(rng.choice(DISTS))


def _windows(torch, X_hi, X_lo, rng):
    """hi and lo as the same window of two larger device matrices: extra
    columns on the right, and a start offset of 0 or 1 element (off the
    16-byte grid)."""
    r, c = X_hi.shape
    off = int(rng.integers(0, 2))
    extra = int(rng.integers(0, 4))
    out = []
    for X in (X_hi, X_lo):
        big = torch.full((r, c + off + extra), 9.0, dtype=torch.float64, device="cuda")
        big[:, off:off + c] = torch.from_numpy(X).cuda()
        out.append(big[:, off:off + c])
    return out


def _bits(x):
    return np.ascontiguousarray(x).view(np.int64)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_strides_and_options(seed):
    import torch
    rng, M, N, K, dist = _case(1000 + seed)
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 2000 + seed)
    t = [*_windows(torch, A_hi, A_lo, rng), *_windows(torch, B_hi, B_lo, rng)]

    R_hi, R_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    C = ddg.dd_gemm(*t)
    assert np.array_equal(_bits(C[0].cpu().numpy()), _bits(R_hi)), (M, N, K, dist)
    assert np.array_equal(_bits(C[1].cpu().numpy()), _bits(R_lo)), (M, N, K, dist)
    KC = -(-K // 8)
    for fs in (False, True):
        for fr in (False, True):
            split_k = int(rng.integers(1, min(KC, 4) + 1)) if not fr else 1
            E = ddg.dd_gemm_ex(*t, split_k=split_k, fuse_split=fs, fuse_recombine=fr)
            assert torch.equal(E[0], C[0]) and torch.equal(E[1], C[1]), (M, N, K, fs, fr, split_k)
    T_hi, T_lo, *_ = slices_bf16.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    T = ddg.dd_gemm_tc(*t)
    assert np.array_equal(_bits(T[0].cpu().numpy()), _bits(T_hi)), (M, N, K, dist)
    assert np.array_equal(_bits(T[1].cpu().numpy()), _bits(T_lo)), (M, N, K, dist)
    assert ddg.wait_timeouts() == 0
