"""The integer-pipe variant of the slice-pair GEMM (int16 parts, exact int64
sums with 32 x 32 -> 64-bit multiply-adds): its parts, its part sums P_d and
its C must equal the oracle's model of the method -- and therefore the FP64
tensor-pipe path -- bit for bit."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices
from tests.gpu_util import dev, host, normwise, special_dd

pytestmark = pytest.mark.gpu

SHAPES = [
    (64, 64, 64, "uniform"),
    (37, 45, 29, "uniform_exp20"),
    (1, 1, 1, "normal"),
    (33, 7, 70, "normal_rowcol30"),
    (5, 96, 200, "uniform"),
    (96, 40, 8, "normal"),
]


def untile_i16(planes, rows, K):
    """planes[((((tile*KC + kc)*8 + kk)*32 + ti)*8) + s] -> D[s, row, k]."""
    Rp = -(-rows // 32) * 32
    Kp = -(-K // 8) * 8
    a = np.asarray(planes).reshape(Rp // 32, Kp // 8, 8, 32, 8)
    return a.transpose(4, 0, 3, 1, 2).reshape(8, Rp, Kp)


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_split_i16_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 5)
    pA, e = ddg.split_rows_i16(dev(A_hi), dev(A_lo))
    pB, f = ddg.split_cols_i16(dev(B_hi), dev(B_lo))
    e_ref, f_ref = slices.row_exponents(A_hi), slices.col_exponents(B_hi)
    assert np.array_equal(host(e), e_ref) and np.array_equal(host(f), f_ref)
    DA = untile_i16(host(pA), M, K)
    DB = untile_i16(host(pB), N, K)
    assert np.array_equal(DA[:, :M, :K], slices.split_rows(A_hi, A_lo, e_ref))
    assert np.array_equal(DB[:, :N, :K], slices.split_cols(B_hi, B_lo, f_ref).transpose(0, 2, 1))
    assert not DA[:, M:, :].any() and not DA[:, :, K:].any()
    assert not DB[:, N:, :].any() and not DB[:, :, K:].any()


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_slice_gemm_i64_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 5)
    pA, _ = ddg.split_rows_i16(dev(A_hi), dev(A_lo))
    pB, _ = ddg.split_cols_i16(dev(B_hi), dev(B_lo))
    DA = slices.split_rows(A_hi, A_lo, slices.row_exponents(A_hi))
    DB = slices.split_cols(B_hi, B_lo, slices.col_exponents(B_hi))
    P_ref = slices.slice_products(DA, DB, exact_int=True)
    KC = -(-K // 8)
    for splits in sorted({s for s in (1, 2, 3, KC) if 1 <= s <= KC}):
        P = host(ddg.slice_gemm_i64(M, N, K, pA, pB, splits))
        Ps = P.sum(axis=0)
        assert np.array_equal(Ps[:, :M, :N], P_ref)
        assert not Ps[:, M:, :].any() and not Ps[:, :, N:].any()
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("M,N,K,dist", SHAPES + [(130, 70, 333, "uniform_exp20"), (300, 260, 1000, "normal")])
def test_dd_gemm_i64_equals_fp64_path_and_model(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 6)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    I_hi, I_lo = ddg.dd_gemm_i64(*t)
    F_hi, F_lo = ddg.dd_gemm(*t)
    I_hi, I_lo, F_hi, F_lo = host(I_hi), host(I_lo), host(F_hi), host(F_lo)
    assert np.array_equal(I_hi.view(np.int64), F_hi.view(np.int64))
    assert np.array_equal(I_lo.view(np.int64), F_lo.view(np.int64))
    if M * N * K <= 10**7:
        M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
        assert np.array_equal(I_hi.view(np.int64), M_hi.view(np.int64))
        assert np.array_equal(I_lo.view(np.int64), M_lo.view(np.int64))
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(I_hi, I_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26


def test_i64_special_values_and_workspace():
    import torch
    rng = np.random.default_rng(16)
    A_hi, A_lo = special_dd(rng, 29, 47)
    B_hi, B_lo = special_dd(rng, 47, 35)
    A_hi[1], A_lo[1] = 0.0, 0.0
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    ws = torch.empty(ddg.workspace_size_i64(29, 35, 47), dtype=torch.uint8, device="cuda")
    I_hi, I_lo = ddg.dd_gemm_i64(*t, workspace=ws)
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(host(I_hi).view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(host(I_lo).view(np.int64), M_lo.view(np.int64))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_i64_workloads(idx):
    import torch
    w = workloads.WORKLOADS[idx]
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    I_hi, I_lo = ddg.dd_gemm_i64(*t)
    torch.cuda.synchronize()
    rng = np.random.default_rng(200 + idx)
    rows = np.unique(np.concatenate([[0, w.M - 1], rng.integers(0, w.M, 4)]))
    cols = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 14)]))
    G_hi = host(I_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(I_lo[torch.from_numpy(rows).cuda()])
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi[rows], A_lo[rows], B_hi[:, cols], B_lo[:, cols])
    assert np.array_equal(G_hi[:, cols].view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo[:, cols].view(np.int64), M_lo.view(np.int64))
    r2 = rows[:2]
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=r2)
    assert normwise(G_hi[:2], G_lo[:2], R_hi, R_lo, A_hi[r2], A_lo[r2], B_hi, B_lo) <= 1e-26
    assert ddg.wait_timeouts() == 0


def test_i64_maximum_k_closed_form():
    import torch
    K = ddg.MAX_K
    A_hi = torch.ones((1, K), dtype=torch.float64, device="cuda")
    A_lo = torch.full((1, K), -2.0**-104, dtype=torch.float64, device="cuda")
    B_hi = torch.ones((K, 1), dtype=torch.float64, device="cuda")
    B_lo = torch.full((K, 1), -2.0**-104, dtype=torch.float64, device="cuda")
    pA, e = ddg.split_rows_i16(A_hi, A_lo)
    pB, f = ddg.split_cols_i16(B_hi, B_lo)
    P = ddg.slice_gemm_i64(1, 1, K, pA, pB, ddg.layout_i64(1, 1, K))
    D = [4095] + [8191] * 7
    P_sum = host(P.sum(dim=0))[:, 0, 0]
    for d in range(8):
        assert P_sum[d] == K * sum(D[s] * D[d - s] for s in range(d + 1))


def test_i64_edge_shapes_and_strides():
    import torch
    # empty products and K = 0
    z = torch.zeros((4, 0), dtype=torch.float64, device="cuda")
    zb = torch.zeros((0, 3), dtype=torch.float64, device="cuda")
    C_hi, C_lo = ddg.dd_gemm_i64(z, z, zb, zb)
    assert C_hi.shape == (4, 3) and not host(C_hi).any() and not np.signbit(host(C_hi)).any()
    e = torch.zeros((0, 5), dtype=torch.float64, device="cuda")
    C_hi, _ = ddg.dd_gemm_i64(e, e, torch.ones((5, 2), dtype=torch.float64, device="cuda"),
                              torch.zeros((5, 2), dtype=torch.float64, device="cuda"))
    assert C_hi.shape == (0, 2)
    # strided, unaligned operands equal the contiguous result
    M, N, K = 19, 23, 37
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 30)
    ref_hi, ref_lo = ddg.dd_gemm_i64(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    big = torch.zeros((M, K + 5), dtype=torch.float64, device="cuda")
    bigl = torch.zeros((M, K + 5), dtype=torch.float64, device="cuda")
    big[:, 1:K + 1], bigl[:, 1:K + 1] = dev(A_hi), dev(A_lo)
    bB = torch.zeros((K, N + 3), dtype=torch.float64, device="cuda")
    bBl = torch.zeros((K, N + 3), dtype=torch.float64, device="cuda")
    bB[:, 1:N + 1], bBl[:, 1:N + 1] = dev(B_hi), dev(B_lo)
    C_hi, C_lo = ddg.dd_gemm_i64(big[:, 1:K + 1], bigl[:, 1:K + 1], bB[:, 1:N + 1], bBl[:, 1:N + 1])
    assert torch.equal(C_hi, ref_hi) and torch.equal(C_lo, ref_lo)


def test_i64_extreme_scales_match_fp64_path():
    M, N, K = 12, 10, 33
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 77)
    ra = np.array([-600, -520, -300, 0, 300, 500, 900, -1000, 1000, 10, -10, 0])
    cb = np.array([-500, -560, 100, 0, -300, 20, 100, 40, -1040, 0])
    A_hi, A_lo = np.ldexp(A_hi, ra[:, None]), np.ldexp(A_lo, ra[:, None])
    B_hi, B_lo = np.ldexp(B_hi, cb[None, :]), np.ldexp(B_lo, cb[None, :])
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    I_hi, I_lo = ddg.dd_gemm_i64(*t)
    F_hi, F_lo = ddg.dd_gemm(*t)
    assert np.array_equal(host(I_hi).view(np.int64), host(F_hi).view(np.int64))
    assert np.array_equal(host(I_lo).view(np.int64), host(F_lo).view(np.int64))
