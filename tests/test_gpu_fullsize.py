"""The full-size workloads, in the launch configuration bench.py times
(dd_gemm_ws with the automatic layout), checked on samples the oracle can
afford: a block of sampled rows x columns bit for bit against the oracle's
model of the method (row / column exponents depend only on that row /
column, so the block is the model's product of the sampled rows and
columns), and whole sampled rows against the exact product (normwise bound
1e-26 on those rows), for the FP64 tensor-pipe path and for the bf16
tensor-core variant.  Plus the maximum inner dimension K = 2^24 with the
largest digits, whose part sums sit just below 2^53 and have a closed form."""
from fractions import Fraction

import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices
from tests.gpu_util import dev, host, normwise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_full_size_workload(idx):
    import torch
    w = workloads.WORKLOADS[idx]
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    tA_hi, tA_lo, tB_hi, tB_lo = dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo)
    ws = torch.empty(ddg.workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device="cuda")
    C_hi, C_lo = ddg.dd_gemm_ws(tA_hi, tA_lo, tB_hi, tB_lo, ws)
    torch.cuda.synchronize()
    assert ddg.wait_timeouts() == 0
    rng = np.random.default_rng(100 + idx)
    rows = np.unique(np.concatenate([[0, w.M // 2, w.M - 1], rng.integers(0, w.M, 3)]))
    cols = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 14)]))
    G_hi = host(C_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(C_lo[torch.from_numpy(rows).cuda()])
    # bit-exact block against the model of the method
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi[rows], A_lo[rows], B_hi[:, cols], B_lo[:, cols])
    assert np.array_equal(G_hi[:, cols].view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo[:, cols].view(np.int64), M_lo.view(np.int64))
    # exact product on two whole rows
    r2 = rows[:2]
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=r2)
    err = normwise(G_hi[:2], G_lo[:2], R_hi, R_lo, A_hi[r2], A_lo[r2], B_hi, B_lo)
    assert err <= 1e-26, err



@pytest.mark.parametrize("idx", [2, 3, 4])
def test_full_size_workload_bf16_variant(idx):
    """The bf16 tensor-core variant (dd_gemm_tc) on the full-size workloads, in
    the layout and k-split bench.py times: a sampled block bit for bit against
    the oracle's model of that variant (13 balanced 8-bit parts, exact sums
    rounded once; the k-splits do not change an exact sum), and two whole
    rows against the exact product."""
    import torch
    from oracle import slices_bf16
    w = workloads.WORKLOADS[idx]
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    ws = torch.empty(ddg.tc_workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device="cuda")
    C_hi = torch.empty((w.M, w.N), dtype=torch.float64, device="cuda")
    C_lo = torch.empty_like(C_hi)
    ddg.dd_gemm_tc(*t, C_hi, C_lo, ws)
    torch.cuda.synchronize()
    assert ddg.wait_timeouts() == 0
    rng = np.random.default_rng(200 + idx)
    rows = np.unique(np.concatenate([[0, w.M // 2, w.M - 1], rng.integers(0, w.M, 3)]))
    cols = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 14)]))
    G_hi = host(C_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(C_lo[torch.from_numpy(rows).cuda()])
    M_hi, M_lo, *_ = slices_bf16.sliced_dd_gemm(A_hi[rows], A_lo[rows], B_hi[:, cols], B_lo[:, cols])
    assert np.array_equal(G_hi[:, cols].view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo[:, cols].view(np.int64), M_lo.view(np.int64))
    r2 = rows[:2]
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=r2)
    err = normwise(G_hi[:2], G_lo[:2], R_hi, R_lo, A_hi[r2], A_lo[r2], B_hi, B_lo)
    assert err <= 1e-26, err

def test_maximum_k_closed_form():
    import torch
    K = ddg.MAX_K
    # x = 1 - 2^-104 as a normalised double double: (1, -2^-104).  With the
    # shared exponent 1, x/2 = 0.0111...1 (104 fraction bits): parts
    # D_0 = 4095 and D_1..7 = 8191, the largest a row can hold.
    A_hi = torch.ones((1, K), dtype=torch.float64, device="cuda")
    A_lo = torch.full((1, K), -2.0**-104, dtype=torch.float64, device="cuda")
    B_hi = torch.ones((K, 1), dtype=torch.float64, device="cuda")
    B_lo = torch.full((K, 1), -2.0**-104, dtype=torch.float64, device="cuda")
    Mp, Np, Kp, splits = ddg.layout(1, 1, K)
    pA, e = ddg.split_rows(A_hi, A_lo)
    pB, f = ddg.split_cols(B_hi, B_lo)
    P = ddg.slice_gemm(1, 1, K, pA, pB, splits)
    D = [4095] + [8191] * 7
    P_sum = host(P.sum(dim=0))[:, 0, 0]
    for d in range(8):
        exact = K * sum(D[s] * D[d - s] for s in range(d + 1))
        assert exact < 2**53
        assert P_sum[d] == exact, (d, P_sum[d], exact)
    del pA, pB
    C_hi, C_lo = ddg.recombine(1, 1, P, e, f)
    assert host(e)[0] == 1 and host(f)[0] == 1
    x = Fraction(1) - Fraction(1, 2**104)
    exact = K * x * x
    got = Fraction(float(host(C_hi)[0, 0])) + Fraction(float(host(C_lo)[0, 0]))
    # per k: truncation of both factors (< 2^-104 each) plus the dropped pairs
    # of index sum 8..14 (sum of (15-d) 2^26 2^(-13(d+2)) < 7.01 2^-104), all
    # times 2^(e+f) = 4; the double-double rounding adds far less
    assert abs(got - exact) <= K * 4 * Fraction(10, 2**104)
    assert got < exact  # truncation toward zero of positive parts
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_full_size_workload_bf16_variant(idx):
    """dd_gemm_tc in the configuration bench.py times: a sampled block bit for bit
    against the oracle's model of the variant, two whole rows against the exact
    product."""
    import torch
    from oracle import slices_bf16
    w = workloads.WORKLOADS[idx]
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    tA_hi, tA_lo, tB_hi, tB_lo = dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo)
    ws = torch.empty(ddg.tc_workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device="cuda")
    C_hi, C_lo = ddg.dd_gemm_tc(tA_hi, tA_lo, tB_hi, tB_lo, workspace=ws)
    torch.cuda.synchronize()
    del ws, tA_hi, tA_lo, tB_hi, tB_lo
    assert ddg.wait_timeouts() == 0
    rng = np.random.default_rng(200 + idx)
    n_rows, n_cols = (3, 4) if w.K > 8192 else (5, 12)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.integers(0, w.M, n_rows - 2)]))
    cols = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, n_cols - 2)]))
    G_hi = host(C_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(C_lo[torch.from_numpy(rows).cuda()])
    M_hi, M_lo, *_ = slices_bf16.sliced_dd_gemm(A_hi[rows], A_lo[rows], B_hi[:, cols], B_lo[:, cols])
    assert np.array_equal(G_hi[:, cols].view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo[:, cols].view(np.int64), M_lo.view(np.int64))
    r2 = rows[:2]
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=r2)
    err = normwise(G_hi[:2], G_lo[:2], R_hi, R_lo, A_hi[r2], A_lo[r2], B_hi, B_lo)
    assert err <= 1e-26, err


def test_bf16_variant_long_k_closed_form():
    """K = 2^20 (128 k-splits of 8192) with x = 1 - 2^-104 everywhere: the part
    sums have the closed form K sum_s D_s D_(d-s) in the int32 planes of every
    split, and C is within the truncation bound of K x^2."""
    import torch
    from oracle import slices_bf16
    K = 1 << 20
    A_hi = torch.ones((1, K), dtype=torch.float64, device="cuda")
    A_lo = torch.full((1, K), -2.0**-104, dtype=torch.float64, device="cuda")
    B_hi = torch.ones((K, 1), dtype=torch.float64, device="cuda")
    B_lo = torch.full((K, 1), -2.0**-104, dtype=torch.float64, device="cuda")
    Mp, Np, Kp, splits = ddg.tc_layout(1, 1, K)
    assert splits >= K // ddg.TC_MAX_K_SPLIT
    pA, e, pB, f = ddg.split_bf16(A_hi, A_lo, B_hi, B_lo)
    assert host(e)[0] == 1 and host(f)[0] == 1          # the parts use e' = 2
    D = slices_bf16.digits_of(1.0, -2.0**-104, 2)
    P = ddg.slice_gemm_tc(1, 1, K, pA, pB, splits)
    del pA, pB
    P_sum = host(P).astype(np.int64).sum(axis=0)[:, 0, 0]
    for d in range(slices_bf16.S):
        assert P_sum[d] == K * sum(D[s] * D[d - s] for s in range(d + 1)), d
    C_hi, C_lo = ddg.recombine_tc(1, 1, P, e, f)
    x = Fraction(1) - Fraction(1, 2**104)
    exact = K * x * x
    got = Fraction(float(host(C_hi)[0, 0])) + Fraction(float(host(C_lo)[0, 0]))
    # per k: truncation of both factors (< 2^-104 each, times 2^(e'+f') = 16)
    # and the dropped pairs (index sums 13..24, < 13 2^14 2^-120 each, times 16)
    assert abs(got - exact) <= K * 16 * Fraction(2 + 13 * 13, 2**104)
    assert ddg.wait_timeouts() == 0


def test_full_size_quad_double_bf16_variant():
    """qd_gemm_tc on the 4096^3 wide-range shape (the quad-double leg bench.py
    times): a sampled block bit for bit against the oracle's model, two whole
    rows within the quad-double gate of the exact product."""
    import torch
    from oracle import slices_bf16_md as bm
    w = workloads.WORKLOADS[2]
    A, B = workloads.make_md(w.M, w.N, w.K, w.dist, w.seed, 4)
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    ws = torch.empty(ddg.qd_tc_workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device="cuda")
    C = ddg.qd_gemm_tc(tA, tB, workspace=ws)
    torch.cuda.synchronize()
    del ws, tA, tB
    assert ddg.wait_timeouts() == 0
    rng = np.random.default_rng(300)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.integers(0, w.M, 1)]))
    cols = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 4)]))
    ridx = torch.from_numpy(rows).cuda()
    G = [host(c[ridx]) for c in C]
    M_ref, *_ = bm.sliced_gemm([a[rows] for a in A], [b[:, cols] for b in B])
    for p in range(4):
        assert np.array_equal(G[p][:, cols].view(np.int64), M_ref[p].view(np.int64)), p
    r2 = rows[:2]
    R = oracle.exact_md_gemm(A, B, rows=r2)
    d = sum(G[p][:2] - R[p] for p in range(4))
    err = float(np.linalg.norm(d) / (np.linalg.norm(sum(a[r2] for a in A)) * np.linalg.norm(sum(B))))
    assert err <= 1e-57, err
