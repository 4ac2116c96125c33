"""Octo (8 doubles, 54 parts) and hexa doubles (16 doubles, 107 parts) with
bf16 parts on the tensor cores (md_gemm_tc): parts, part sums and every plane
of C bit for bit against the oracle's model (oracle.slices_bf16_md), and C
within the normwise gate of the exact multiple-double product (2^-404 /
2^-828, measured with exact rational differences)."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices_bf16_md as bm
from tests.gpu_util import dev, host
from tests.test_gpu_tc import pad, unswizzle
from tests.test_oracle_bf16_md import log2_normwise

pytestmark = pytest.mark.gpu

CASES = [(8, -404), (16, -828)]  # doubles per number, log2 of the gate
SHAPES = [(9, 7, 21, "uniform_exp20"), (1, 1, 1, "normal"), (40, 30, 70, "normal_rowcol30")]


@pytest.mark.parametrize("n,gate", CASES)
@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_md_tc_parts_and_product(n, gate, M, N, K, dist):
    S = ddg.MD_TC_PARTS[n]
    A, B = workloads.make_md(M, N, K, dist, 5 + n, n)
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    C_ref, e_ref, f_ref, DA, DB, P_ref = bm.sliced_gemm(A, B, S)
    pA, e, pB, f = ddg.md_split_bf16(tA, tB)
    assert np.array_equal(host(e) + 1, e_ref) and np.array_equal(host(f) + 1, f_ref)
    GA = unswizzle(host(pA), pad(M, ddg.TC_TILE_M), K, ddg.TC_BLOCK_M, parts=S)
    GB = unswizzle(host(pB), pad(N, ddg.TC_TILE_N), K, ddg.TC_TILE_N, parts=S)
    assert np.array_equal(GA[:, :M, :K], DA)
    assert np.array_equal(GB[:, :N, :K], DB.transpose(0, 2, 1))
    sp = ddg.md_tc_layout(n, M, N, K)[3]
    P = ddg.md_slice_gemm_tc(n, M, N, K, pA, pB, sp)
    assert np.array_equal(host(P).astype(np.int64).sum(axis=0)[:, :M, :N], P_ref)
    Cr = [host(c) for c in ddg.md_recombine_tc(n, M, N, P, e, f)]
    C = [host(c) for c in ddg.md_gemm_tc(tA, tB)]
    for p in range(n):
        assert np.array_equal(Cr[p].view(np.int64), C_ref[p].view(np.int64)), p
        assert np.array_equal(C[p].view(np.int64), C_ref[p].view(np.int64)), p
    R = oracle.exact_md_gemm(A, B)
    assert log2_normwise(C, R, A, B) <= gate
    assert ddg.wait_timeouts() == 0


def test_md_tc_k_splits_and_errors():
    # K = 1100 > 1024: hexa doubles need two k-splits
    n, M, N, K = 16, 3, 4, 1100
    A, B = workloads.make_md(M, N, K, "uniform", 9, n)
    Mp, Np, Kp, sp = ddg.md_tc_layout(n, M, N, K)
    assert sp >= 2
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    pA, e, pB, f = ddg.md_split_bf16(tA, tB)
    with pytest.raises(ddg.DDGemmError):
        ddg.md_slice_gemm_tc(n, M, N, K, pA, pB, 1)
    C = [host(c) for c in ddg.md_gemm_tc(tA, tB)]
    R = oracle.exact_md_gemm(A, B)
    assert log2_normwise(C, R, A, B) <= -828
    lib = ddg.load()
    assert lib.md_gemm_tc(4, 2, 2, 2, None, 2, None, 2, None, 2, None, 0, None) == 2  # quad doubles: qd_gemm_tc
    assert ddg.wait_timeouts() == 0


def test_md_tc_tiny_values_round_with_gradual_underflow():
    # octo doubles near the bottom of the exponent range: the lower parts of
    # the product are subnormal or zero, as in the exact oracle's expansion
    n = 8
    A, B = workloads.make_md(5, 4, 9, "uniform", 11, n)
    A = [a * 2.0**-480 for a in A]
    B = [b * 2.0**-470 for b in B]
    C = [host(c) for c in ddg.md_gemm_tc([dev(a) for a in A], [dev(b) for b in B])]
    C_ref, *_ = bm.sliced_gemm(A, B, ddg.MD_TC_PARTS[n])
    for p in range(n):
        assert np.array_equal(C[p].view(np.int64), C_ref[p].view(np.int64)), p
    assert ddg.wait_timeouts() == 0


def _md_digits_of_sum(Z, S_):
    s, a = (-1, -Z) if Z < 0 else (1, Z)
    top = 8 * (S_ - 1)
    return [s * (a >> top)] + [s * ((a >> (8 * (S_ - 1 - d))) & 0xFF) for d in range(1, S_)]


@pytest.mark.parametrize("n", [8, 16])
def test_md_recombine_rounding_cases(n):
    """Crafted and random exact sums against the oracle's rounding into n
    doubles: ties (to even, both ways) in the first, a middle and the last
    part, long runs of ones and zeros (remainders that flip sign part after
    part), both signs, small values, zero, and scales at the ends of the
    normal range (q = -1022 and -1023); then random int32 part sums."""
    S_ = ddg.MD_TC_PARTS[n]
    top = 8 * (S_ - 1) + 28                       # |Z| < 2^top keeps v_0 in int32
    crafted = [
        (2**52 + 1) * 2**(top - 60) + 2**(top - 61),                  # tie in x0, odd
        2**52 * 2**(top - 60) + 2**(top - 61),                        # tie in x0, even
        2**top - 1,                                                   # ones: every part rounds up
        2**top - 2**(top // 2) + 1,
        2**(top - 2) + (2**52 + 1) * 2**(top - 150) + 2**(top - 151),  # tie in x1
        2**(top - 2) + 2**(top - 70) + 2**(top - 140) + (2**52 + 1) * 2**60 + 2**59,
        sum(2**(top - 2 - 57 * k) for k in range(n)) + 2**3,           # one bit per part
        (2**52 + 1) * 2 + 1, 12345, 1, 0,
    ]
    crafted += [-z for z in crafted if z]
    rng = np.random.default_rng(30 + n)
    # q = e + f + 2 - 8 (S + 1): -1022 and -1023 at f = 0, and large scales
    base = 8 * (S_ + 1) - 2
    E = [0, -1022 + base, -1023 + base, 300, 1022 - top + base - 2, -900]
    M, Nc, Nr = len(E), len(crafted), 100
    N = Nc + Nr
    Mp, Np = pad(M, ddg.TC_TILE_M), pad(N, ddg.TC_TILE_N)
    e = np.array(E, dtype=np.int32)
    f = np.concatenate([np.zeros(Nc), rng.integers(-6, 7, Nr)]).astype(np.int32)
    for splits in (1, 2):
        P = np.zeros((splits, S_, Mp, Np), dtype=np.int32)
        for c, Z in enumerate(crafted):
            P[0, :, :M, c] = np.array(_md_digits_of_sum(Z, S_), dtype=np.int64)[:, None]
        lim = np.iinfo(np.int32)
        P[:, :, :M, Nc:N] = rng.integers(lim.min, lim.max, (splits, S_, M, Nr), endpoint=True)
        R = bm.recombine(P.astype(np.int64).sum(axis=0)[:, :M, :N], e + 1, f + 1, n)
        C = [host(c) for c in ddg.md_recombine_tc(n, M, N, dev(P), dev(e), dev(f))]
        for p in range(n):
            assert np.array_equal(C[p].view(np.int64), R[p].view(np.int64)), (splits, p)
    assert ddg.wait_timeouts() == 0
