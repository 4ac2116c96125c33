"""GPU path vs the oracle, through the C ABI, at sizes the oracle finishes in
seconds.  Integer work (exponents, 13-bit parts, slice-pair sums) must match
bit for bit; the recombination follows the same round-to-nearest sequence as
the oracle's model and must match bit for bit too; the product must be within
the normwise bound 1e-26 of the exact product."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices
from tests.gpu_util import dev, host, normwise, special_dd, untile

pytestmark = pytest.mark.gpu

SHAPES = [
    (64, 64, 64, "uniform"),
    (37, 45, 29, "uniform_exp20"),
    (1, 1, 1, "normal"),
    (33, 7, 70, "normal_rowcol30"),
    (5, 96, 200, "uniform"),
    (96, 40, 8, "normal"),
]


def _inputs(M, N, K, dist, seed=5):
    return workloads.make_dd(M, N, K, dist, seed)


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_split_rows_bit_exact(M, N, K, dist):
    A_hi, A_lo, _, _ = _inputs(M, N, K, dist)
    planes, e = ddg.split_rows(dev(A_hi), dev(A_lo))
    e_ref = slices.row_exponents(A_hi)
    D_ref = slices.split_rows(A_hi, A_lo, e_ref)
    assert np.array_equal(host(e), e_ref)
    D = untile(host(planes), M, K)
    assert np.array_equal(D[:, :M, :K], D_ref.astype(np.float64))
    assert not D[:, M:, :].any() and not D[:, :, K:].any()


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_split_cols_bit_exact(M, N, K, dist):
    _, _, B_hi, B_lo = _inputs(M, N, K, dist)
    planes, f = ddg.split_cols(dev(B_hi), dev(B_lo))
    f_ref = slices.col_exponents(B_hi)
    D_ref = slices.split_cols(B_hi, B_lo, f_ref)
    assert np.array_equal(host(f), f_ref)
    D = untile(host(planes), N, K)  # D[t, j, k]
    assert np.array_equal(D[:, :N, :K], D_ref.transpose(0, 2, 1).astype(np.float64))
    assert not D[:, N:, :].any() and not D[:, :, K:].any()


def test_split_special_values():
    rng = np.random.default_rng(9)
    A_hi, A_lo = special_dd(rng, 40, 51)
    A_hi[3] = 0.0
    A_lo[3] = 0.0            # an all-zero row: exponent 0, all parts 0
    planes, e = ddg.split_rows(dev(A_hi), dev(A_lo))
    e_ref = slices.row_exponents(A_hi)
    assert np.array_equal(host(e), e_ref) and e_ref[3] == 0
    D = untile(host(planes), 40, 51)[:, :40, :51]
    assert np.array_equal(D, slices.split_rows(A_hi, A_lo, e_ref).astype(np.float64))
    B_hi, B_lo = special_dd(rng, 51, 33)
    B_hi[:, 5] = 0.0
    B_lo[:, 5] = 0.0
    planes, f = ddg.split_cols(dev(B_hi), dev(B_lo))
    f_ref = slices.col_exponents(B_hi)
    assert np.array_equal(host(f), f_ref)
    D = untile(host(planes), 33, 51)[:, :33, :51]
    assert np.array_equal(D, slices.split_cols(B_hi, B_lo, f_ref).transpose(0, 2, 1).astype(np.float64))


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_slice_gemm_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, dist)
    pA, e = ddg.split_rows(dev(A_hi), dev(A_lo))
    pB, f = ddg.split_cols(dev(B_hi), dev(B_lo))
    DA = slices.split_rows(A_hi, A_lo, slices.row_exponents(A_hi))
    DB = slices.split_cols(B_hi, B_lo, slices.col_exponents(B_hi))
    P_ref = slices.slice_products(DA, DB)
    KC = -(-K // 8)
    for splits in sorted({s for s in (1, 2, 3, KC) if 1 <= s <= KC}):
        P = host(ddg.slice_gemm(M, N, K, pA, pB, splits))
        assert P.shape[0] == splits
        Ps = P.sum(axis=0)  # integers below 2^53: exact
        assert np.array_equal(Ps[:, :M, :N], P_ref)
        assert not Ps[:, M:, :].any() and not Ps[:, :, N:].any()
        # each split is the same sum over its own k-chunks
        z = splits - 1
        k0, k1 = z * KC // splits * 8, min(K, (z + 1) * KC // splits * 8)
        P_z = slices.slice_products(DA[:, :, k0:k1], DB[:, k0:k1, :])
        assert np.array_equal(P[z][:, :M, :N], P_z)


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_recombine_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, dist)
    C_ref_hi, C_ref_lo, e_ref, f_ref, DA, DB, P_ref = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    pA, e = ddg.split_rows(dev(A_hi), dev(A_lo))
    pB, f = ddg.split_cols(dev(B_hi), dev(B_lo))
    P = ddg.slice_gemm(M, N, K, pA, pB, 1)
    C_hi, C_lo = ddg.recombine(M, N, P, e, f)
    assert np.array_equal(host(C_hi).view(np.int64), C_ref_hi.view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), C_ref_lo.view(np.int64))


@pytest.mark.parametrize("M,N,K,dist", SHAPES + [(130, 70, 333, "uniform_exp20")])
def test_dd_gemm_matches_model_and_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, dist)
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    C_hi, C_lo = host(C_hi), host(C_lo)
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(C_hi.view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(C_lo.view(np.int64), M_lo.view(np.int64))
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("idx", [0, 1])
def test_small_workloads_full_check(idx):
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    C_hi, C_lo = host(C_hi), host(C_lo)
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    err = normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo)
    assert err <= 1e-26, err
    # bit-exact against the model of the method
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(C_hi.view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(C_lo.view(np.int64), M_lo.view(np.int64))


def test_special_values_end_to_end():
    rng = np.random.default_rng(10)
    A_hi, A_lo = special_dd(rng, 23, 41)
    B_hi, B_lo = special_dd(rng, 41, 19)
    A_hi[2], A_lo[2] = 0.0, 0.0
    B_hi[:, 3], B_lo[:, 3] = 0.0, 0.0
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(host(C_hi).view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), M_lo.view(np.int64))
    assert not np.signbit(host(C_hi)[2]).any() and not host(C_hi)[2].any()


def test_empty_and_zero_k():
    import torch
    z = torch.zeros((4, 0), dtype=torch.float64, device="cuda")
    zb = torch.zeros((0, 3), dtype=torch.float64, device="cuda")
    C_hi, C_lo = ddg.dd_gemm(z, z, zb, zb)
    assert C_hi.shape == (4, 3)
    assert not host(C_hi).any() and not host(C_lo).any()
    assert not np.signbit(host(C_hi)).any()
    e = torch.zeros((0, 5), dtype=torch.float64, device="cuda")
    C_hi, C_lo = ddg.dd_gemm(e, e, torch.ones((5, 2), dtype=torch.float64, device="cuda"),
                             torch.zeros((5, 2), dtype=torch.float64, device="cuda"))
    assert C_hi.shape == (0, 2)


def test_strided_and_unaligned_inputs():
    import torch
    M, N, K = 19, 23, 37
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, "normal")
    ref_hi, ref_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    # leading dimensions larger than the width, and base pointers offset by one
    # double (not 16-byte aligned: the scalar-load paths)
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
    C_hi, C_lo = ddg.dd_gemm(big[:, 1:K + 1], bigl[:, 1:K + 1], bB[:, 1:N + 1], bBl[:, 1:N + 1],
                             Cb[:, 2:N + 2], Cl[:, 2:N + 2])
    assert torch.equal(C_hi, ref_hi) and torch.equal(C_lo, ref_lo)
    # the output's padding columns are untouched
    assert torch.all(Cb[:, :2] == 7.0) and torch.all(Cb[:, N + 2:] == 7.0)


def test_variants_and_determinism():
    import torch
    M, N, K = 70, 45, 300
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, "uniform_exp20")
    tA_hi, tA_lo, tB_hi, tB_lo = dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo)
    C1 = ddg.dd_gemm(tA_hi, tA_lo, tB_hi, tB_lo)
    C2 = ddg.dd_gemm(tA_hi, tA_lo, tB_hi, tB_lo)
    assert torch.equal(C1[0], C2[0]) and torch.equal(C1[1], C2[1])
    ws = torch.empty(ddg.workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    C3 = ddg.dd_gemm_ws(tA_hi, tA_lo, tB_hi, tB_lo, ws)
    assert torch.equal(C1[0], C3[0]) and torch.equal(C1[1], C3[1])
    H_hi = np.zeros((M, N))
    H_lo = np.zeros((M, N))
    ddg.dd_gemm_host(A_hi, A_lo, B_hi, B_lo, H_hi, H_lo)
    assert np.array_equal(H_hi, host(C1[0])) and np.array_equal(H_lo, host(C1[1]))
    # on another stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C4 = ddg.dd_gemm(tA_hi, tA_lo, tB_hi, tB_lo)
    s.synchronize()
    assert torch.equal(C1[0], C4[0]) and torch.equal(C1[1], C4[1])


def test_identity_returns_truncated_parts():
    # A * I: each output is the 8-part truncation of A's element on its row
    # grid, recombined; for plain doubles (lo = 0) that is A itself.
    rng = np.random.default_rng(12)
    M, K = 21, 40
    A_hi = rng.normal(size=(M, K)) * np.ldexp(1.0, rng.integers(-10, 10, (M, 1)))
    A_lo = np.zeros_like(A_hi)
    I = np.eye(K)
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(I), dev(np.zeros_like(I)))
    # row exponents span at most ~2^20 inside a row here, so 104 bits hold every double
    assert np.array_equal(host(C_hi), A_hi) and not host(C_lo).any()


def test_no_wait_timeouts():
    assert ddg.wait_timeouts() == 0


def test_extreme_scales_match_model():
    # rows and columns scaled towards the ends of the exponent range: shared
    # exponents near +-1000, products that land in the subnormal range and
    # near the overflow threshold; the GPU must follow the model bit for bit
    # (including the correctly rounded final scaling)
    rng = np.random.default_rng(13)
    M, N, K = 12, 10, 33
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 77)
    ra = np.array([-600, -520, -300, 0, 300, 500, 900, -1000, 1000, 10, -10, 0])
    cb = np.array([-500, -560, 100, 0, -300, 20, 100, 40, -1040, 0])
    A_hi, A_lo = np.ldexp(A_hi, ra[:, None]), np.ldexp(A_lo, ra[:, None])
    B_hi, B_lo = np.ldexp(B_hi, cb[None, :]), np.ldexp(B_lo, cb[None, :])
    assert np.all(np.isfinite(A_lo)) and np.all(np.isfinite(B_lo))
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(host(C_hi).view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), M_lo.view(np.int64))
    # entries whose scale stays in the normal range are within the bound of
    # the exact product, entry by entry relative to |A||B|
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    mag = np.abs(A_hi) @ np.abs(B_hi)
    ok = (mag > 2.0**-900) & (mag < 2.0**900)
    err = np.abs((host(C_hi) - R_hi) + (host(C_lo) - R_lo))
    assert np.all(err[ok] <= 1e-28 * mag[ok])


def test_many_row_tiles():
    # more than 65535 row tiles (a grid-dimension limit the kernels must not
    # inherit) and a ragged last tile
    import torch
    M, N, K = 65536 * 32 + 7, 40, 24
    rng = np.random.default_rng(14)
    A_hi = rng.uniform(-1, 1, (M, K))
    A_lo = A_hi * 2.0**-54 * rng.uniform(-1, 1, (M, K))
    s = A_hi + A_lo
    A_lo = A_lo - (s - A_hi)
    A_hi = s
    _, _, B_hi, B_lo = workloads.make_dd(1, N, K, "uniform", 15)
    C_hi, C_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    rows = np.array([0, 1, 31, 32, M // 2, M - 33, M - 1])
    G_hi = host(C_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(C_lo[torch.from_numpy(rows).cuda()])
    M_hi, M_lo, *_ = slices.sliced_dd_gemm(A_hi[rows], A_lo[rows], B_hi, B_lo)
    assert np.array_equal(G_hi.view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo.view(np.int64), M_lo.view(np.int64))


@pytest.mark.parametrize("M,N,K,dist", SHAPES[:4])
def test_combined_split_equals_separate(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = _inputs(M, N, K, dist)
    t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
    pA, e, pB, f = ddg.split(*t)
    qA, e2 = ddg.split_rows(t[0], t[1])
    qB, f2 = ddg.split_cols(t[2], t[3])
    assert torch_equal(pA, qA) and torch_equal(pB, qB) and torch_equal(e, e2) and torch_equal(f, f2)
    iA, ie, iB, jf = ddg.split_i16(*t)
    rA, re_ = ddg.split_rows_i16(t[0], t[1])
    rB, rf = ddg.split_cols_i16(t[2], t[3])
    assert torch_equal(iA, rA) and torch_equal(iB, rB) and torch_equal(ie, re_) and torch_equal(jf, rf)


def torch_equal(a, b):
    import torch
    return bool(torch.equal(a, b))
