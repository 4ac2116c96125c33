"""The split fused into the slice GEMM's prologue and the recombination fused
into its epilogue (dd_gemm_ex, dd_slice_gemm_fused), through the C ABI.

The fused GEMM forms the same 13-bit parts as the split kernel, so its part
sums P must equal the oracle model's slice-pair sums bit for bit; every
option combination of dd_gemm_ex must give the model's C bit for bit (and
dd_gemm's), and stay within the normwise bound of the exact product."""
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
    (130, 70, 333, "uniform_exp20"),
]

COMBOS = [(fs, fr) for fs in (False, True) for fr in (False, True)]


def _bits(x):
    return np.ascontiguousarray(x).view(np.int64)


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_fused_slice_gemm_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 41)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    e, f = ddg.exponents(t[0], t[2])
    DA = slices.split_rows(A_hi, A_lo, slices.row_exponents(A_hi))
    DB = slices.split_cols(B_hi, B_lo, slices.col_exponents(B_hi))
    P_ref = slices.slice_products(DA, DB)
    KC = -(-K // 8)
    for splits in sorted({s for s in (1, 2, 3, KC) if 1 <= s <= KC}):
        P = host(ddg.slice_gemm_fused(*t, e, f, splits))
        Ps = P.sum(axis=0)  # integers below 2^53: exact
        assert np.array_equal(Ps[:, :M, :N], P_ref)
        assert not Ps[:, M:, :].any() and not Ps[:, :, N:].any()
        z = splits - 1
        k0, k1 = z * KC // splits * 8, min(K, (z + 1) * KC // splits * 8)
        assert np.array_equal(P[z][:, :M, :N], slices.slice_products(DA[:, :, k0:k1], DB[:, k0:k1, :]))


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
@pytest.mark.parametrize("fuse_split,fuse_recombine", COMBOS)
def test_dd_gemm_ex_matches_model(M, N, K, dist, fuse_split, fuse_recombine):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 42)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    KC = -(-K // 8)
    splits_to_try = [0, 1] + ([2, 3] if not fuse_recombine and KC >= 3 else [])
    for split_k in splits_to_try:
        C_hi, C_lo = ddg.dd_gemm_ex(*t, split_k=split_k, fuse_split=fuse_split, fuse_recombine=fuse_recombine)
        assert np.array_equal(_bits(host(C_hi)), _bits(M_hi)), split_k
        assert np.array_equal(_bits(host(C_lo)), _bits(M_lo)), split_k
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(host(C_hi), host(C_lo), R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("fuse_split,fuse_recombine", COMBOS)
def test_ex_special_values(fuse_split, fuse_recombine):
    rng = np.random.default_rng(43)
    A_hi, A_lo = special_dd(rng, 23, 41)
    B_hi, B_lo = special_dd(rng, 41, 19)
    A_hi[2], A_lo[2] = 0.0, 0.0
    B_hi[:, 3], B_lo[:, 3] = 0.0, 0.0
    C_hi, C_lo = ddg.dd_gemm_ex(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo), split_k=1, fuse_split=fuse_split,
                                fuse_recombine=fuse_recombine)
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(_bits(host(C_hi)), _bits(M_hi))
    assert np.array_equal(_bits(host(C_lo)), _bits(M_lo))
    assert not np.signbit(host(C_hi)[2]).any() and not host(C_hi)[2].any()


@pytest.mark.parametrize("fuse_split,fuse_recombine", COMBOS)
def test_ex_extreme_scales(fuse_split, fuse_recombine):
    # shared exponents near +-1000 and results in the subnormal range: the
    # epilogue's final scaling must round as the recombine kernel's does
    M, N, K = 12, 10, 33
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 77)
    ra = np.array([-600, -520, -300, 0, 300, 500, 900, -1000, 1000, 10, -10, 0])
    cb = np.array([-500, -560, 100, 0, -300, 20, 100, 40, -1040, 0])
    A_hi, A_lo = np.ldexp(A_hi, ra[:, None]), np.ldexp(A_lo, ra[:, None])
    B_hi, B_lo = np.ldexp(B_hi, cb[None, :]), np.ldexp(B_lo, cb[None, :])
    C_hi, C_lo = ddg.dd_gemm_ex(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo), split_k=1, fuse_split=fuse_split,
                                fuse_recombine=fuse_recombine)
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(_bits(host(C_hi)), _bits(M_hi))
    assert np.array_equal(_bits(host(C_lo)), _bits(M_lo))


@pytest.mark.parametrize("fuse_split,fuse_recombine", COMBOS)
def test_ex_strided_unaligned_and_padding(fuse_split, fuse_recombine):
    import torch
    M, N, K = 19, 23, 37
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 44)
    ref_hi, ref_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    big = torch.zeros((M, K + 5), dtype=torch.float64, device="cuda")
    bigl = torch.zeros((M, K + 5), dtype=torch.float64, device="cuda")
    big[:, 1:K + 1] = dev(A_hi)
    bigl[:, 1:K + 1] = dev(A_lo)
    bB = torch.zeros((K, N + 3), dtype=torch.float64, device="cuda")
    bBl = torch.zeros((K, N + 3), dtype=torch.float64, device="cuda")
    bB[:, 1:N + 1] = dev(B_hi)
    bBl[:, 1:N + 1] = dev(B_lo)
    Cb = torch.full((M, N + 4), 7.0, dtype=torch.float64, device="cuda")
    Cl = torch.full((M, N + 4), 7.0, dtype=torch.float64, device="cuda")
    C_hi, C_lo = ddg.dd_gemm_ex(big[:, 1:K + 1], bigl[:, 1:K + 1], bB[:, 1:N + 1], bBl[:, 1:N + 1],
                                Cb[:, 2:N + 2], Cl[:, 2:N + 2], split_k=1, fuse_split=fuse_split,
                                fuse_recombine=fuse_recombine)
    assert torch.equal(C_hi, ref_hi) and torch.equal(C_lo, ref_lo)
    assert torch.all(Cb[:, :2] == 7.0) and torch.all(Cb[:, N + 2:] == 7.0)
    assert torch.all(Cl[:, :2] == 7.0) and torch.all(Cl[:, N + 2:] == 7.0)
    # aligned lda, odd ldc (scalar stores in the fused epilogue)
    Co = torch.full((M, N + 1), 7.0, dtype=torch.float64, device="cuda")
    Col = torch.full((M, N + 1), 7.0, dtype=torch.float64, device="cuda")
    ddg.dd_gemm_ex(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo), Co[:, :N], Col[:, :N], split_k=1,
                   fuse_split=fuse_split, fuse_recombine=fuse_recombine)
    assert torch.equal(Co[:, :N], ref_hi) and torch.equal(Col[:, :N], ref_lo)
    assert torch.all(Co[:, N] == 7.0) and torch.all(Col[:, N] == 7.0)


@pytest.mark.parametrize("fuse_split,fuse_recombine", COMBOS)
def test_ex_empty_and_zero_k(fuse_split, fuse_recombine):
    import torch
    z = torch.zeros((4, 0), dtype=torch.float64, device="cuda")
    zb = torch.zeros((0, 3), dtype=torch.float64, device="cuda")
    C_hi, C_lo = ddg.dd_gemm_ex(z, z, zb, zb, fuse_split=fuse_split, fuse_recombine=fuse_recombine)
    assert C_hi.shape == (4, 3)
    assert not host(C_hi).any() and not host(C_lo).any() and not np.signbit(host(C_hi)).any()
    e = torch.zeros((0, 5), dtype=torch.float64, device="cuda")
    C_hi, _ = ddg.dd_gemm_ex(e, e, torch.ones((5, 2), dtype=torch.float64, device="cuda"),
                             torch.zeros((5, 2), dtype=torch.float64, device="cuda"),
                             fuse_split=fuse_split, fuse_recombine=fuse_recombine)
    assert C_hi.shape == (0, 2)


def test_ex_workspace_and_plan():
    import torch
    M, N, K = 300, 260, 1000
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "uniform_exp20", 45)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    ref = ddg.dd_gemm(*t)
    for fs, fr in COMBOS:
        nbytes, splits, fused = ddg.ex_plan(M, N, K, split_k=1, fuse_split=fs, fuse_recombine=fr)
        assert splits == 1 and fused == fr
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        C = ddg.dd_gemm_ex(*t, split_k=1, fuse_split=fs, fuse_recombine=fr, workspace=ws)
        assert torch.equal(C[0], ref[0]) and torch.equal(C[1], ref[1])
    # both fusions: the workspace holds only the exponents
    nbytes, _, _ = ddg.ex_plan(M, N, K, split_k=1, fuse_split=True, fuse_recombine=True)
    assert nbytes == 1280 + 1280  # e (320 int32) and f (288 int32), each 256-byte aligned


def test_ex_two_calls_in_a_row_and_streams():
    import torch
    M, N, K = 70, 45, 300
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "uniform_exp20", 46)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    ref = ddg.dd_gemm(*t)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C1 = ddg.dd_gemm_ex(*t, fuse_split=True, fuse_recombine=True)
        C2 = ddg.dd_gemm_ex(*t, fuse_split=True, fuse_recombine=True)
    s.synchronize()
    for C in (C1, C2):
        assert torch.equal(C[0], ref[0]) and torch.equal(C[1], ref[1])
