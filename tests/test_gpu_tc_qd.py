"""Quad doubles with 27 bf16 parts on the tensor cores (qd_gemm_tc): parts,
part sums and the four planes of C bit for bit against the oracle's model
(oracle.slices_bf16_md), and C within the quad-double gate of the exact
multiple-double product."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices_bf16_md as bm
from tests.gpu_util import dev, host
from tests.test_gpu_tc import pad, unswizzle

pytestmark = pytest.mark.gpu

QD_GATE = 1e-57
S = bm.QD_PARTS
SHAPES = [
    (64, 64, 64, "uniform"),
    (37, 45, 29, "uniform_exp20"),
    (1, 1, 1, "normal"),
    (130, 260, 130, "normal_rowcol30"),
]


def _qd_normwise(C, R, A, B):
    d = sum(C[p] - R[p] for p in range(4))
    return float(np.linalg.norm(d) / (np.linalg.norm(sum(A)) * np.linalg.norm(sum(B))))


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_qd_split_bf16_bit_exact(M, N, K, dist):
    A, B = workloads.make_md(M, N, K, dist, 3, 4)
    pA, e, pB, f = ddg.qd_split_bf16([dev(a) for a in A], [dev(b) for b in B])
    e_ref, f_ref = bm.row_exponents(A[0]), bm.col_exponents(B[0])
    assert np.array_equal(host(e) + 1, e_ref) and np.array_equal(host(f) + 1, f_ref)
    DA = unswizzle(host(pA), pad(M, ddg.TC_TILE_M), K, ddg.TC_BLOCK_M, parts=S)
    DB = unswizzle(host(pB), pad(N, ddg.TC_TILE_N), K, ddg.TC_TILE_N, parts=S)
    assert np.array_equal(DA[:, :M, :K], bm.split_rows(A, e_ref, S))
    assert np.array_equal(DB[:, :N, :K], bm.split_cols(B, f_ref, S).transpose(0, 2, 1))
    assert not DA[:, M:, :].any() and not DA[:, :, K:].any()


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_qd_gemm_tc_steps_and_whole(M, N, K, dist):
    A, B = workloads.make_md(M, N, K, dist, 4, 4)
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    C_ref, e_ref, f_ref, DA, DB, P_ref = bm.sliced_gemm(A, B)
    pA, e, pB, f = ddg.qd_split_bf16(tA, tB)
    KB = -(-K // 64)
    for splits in sorted({s for s in (1, 2, KB) if 1 <= s <= KB}):
        P = host(ddg.qd_slice_gemm_tc(M, N, K, pA, pB, splits)).astype(np.int64)
        assert np.array_equal(P.sum(axis=0)[:, :M, :N], P_ref), splits
        Cr = [host(c) for c in ddg.qd_recombine_tc(M, N, ddg.qd_slice_gemm_tc(M, N, K, pA, pB, splits), e, f)]
        for p in range(4):
            assert np.array_equal(Cr[p].view(np.int64), C_ref[p].view(np.int64)), (splits, p)
    C = [host(c) for c in ddg.qd_gemm_tc(tA, tB)]
    for p in range(4):
        assert np.array_equal(C[p].view(np.int64), C_ref[p].view(np.int64)), p
    R = oracle.exact_md_gemm(A, B)
    assert _qd_normwise(C, R, A, B) <= QD_GATE
    assert ddg.wait_timeouts() == 0


def test_qd_gemm_tc_k_split_bound_and_errors():
    # K = 4100 > 4096: two k-splits of at most 4096, exact int32 sums
    M, N, K = 3, 5, 4100
    A, B = workloads.make_md(M, N, K, "normal", 6, 4)
    Mp, Np, Kp, sp = ddg.qd_tc_layout(M, N, K)
    assert sp >= 2 and -(-(Kp // 64) // sp) * 64 <= ddg.TC_QD_MAX_K_SPLIT
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    pA, e, pB, f = ddg.qd_split_bf16(tA, tB)
    with pytest.raises(ddg.DDGemmError):
        ddg.qd_slice_gemm_tc(M, N, K, pA, pB, 1)
    C = [host(c) for c in ddg.qd_gemm_tc(tA, tB)]
    R = oracle.exact_md_gemm(A, B)
    assert _qd_normwise(C, R, A, B) <= QD_GATE
    lib = ddg.load()
    assert lib.qd_gemm_tc(2, 2, ddg.QD_MAX_K + 1, None, ddg.QD_MAX_K + 1, None, 2, None, 2, None, 0, None) == 2
    assert ddg.wait_timeouts() == 0


def _qd_digits_of_sum(Z):
    """27 part sums whose exact sum sum_d v_d 256^(26-d) is Z (v_0 = the bits
    above 208, base-256 digits below; negated for a negative Z)."""
    s, a = (-1, -Z) if Z < 0 else (1, Z)
    return [s * (a >> 208)] + [s * ((a >> (8 * (26 - d))) & 0xFF) for d in range(1, S)]


def test_qd_recombine_rounding_cases():
    """Crafted part sums against the oracle's rounding into four doubles: a
    tie in each of the four (to even, either way), carries to the next power
    of two, remainders of both signs, exact small values, zero, both signs and
    scales at the ends of the normal range; then random int32 part sums with
    one and two k-splits."""
    crafted = [
        (2**52 + 1) * 2**180 + 2**179,                       # tie in x0, odd: up
        2**52 * 2**180 + 2**179,                             # tie in x0, even: down
        (2**53 + 1) * 2**180 + 2**179,                       # above half an ulp
        2**236 + (2**52 + 1) * 2**100 + 2**99,               # tie in x1
        2**236 + 2**170 + (2**52 + 1) * 2**50 + 2**49,       # tie in x2
        2**236 + 2**170 + 2**110 + (2**52 + 1) * 4 + 2,      # tie in x3
        2**236 + 2**170 + 2**110 + 2**52 * 4 + 2,            # tie in x3, even
        2**237 - 1,                                          # carries all the way up
        2**236 - 2**100 + 3,                                 # remainders change sign
        (2**53 - 1) * 2**150 + 2**149 + 1,                   # rounds up to 2^203
        12345, 1, 0,
    ]
    crafted += [-z for z in crafted if z]
    rng = np.random.default_rng(22)
    E = [0, -800, -801, 700, 1000, 1010, -990]  # q = e + f - 222: -1022 and -1023 at f = 0
    M, Nc, Nr = len(E), len(crafted), 150
    N = Nc + Nr
    Mp, Np = pad(M, ddg.TC_TILE_M), pad(N, ddg.TC_TILE_N)
    e = np.array(E, dtype=np.int32)
    f = np.concatenate([np.zeros(Nc), rng.integers(-6, 7, Nr)]).astype(np.int32)
    for splits in (1, 2):
        P = np.zeros((splits, S, Mp, Np), dtype=np.int32)
        for c, Z in enumerate(crafted):
            P[0, :, :M, c] = np.array(_qd_digits_of_sum(Z), dtype=np.int64)[:, None]
        lim = np.iinfo(np.int32)
        P[:, :, :M, Nc:N] = rng.integers(lim.min, lim.max, (splits, S, M, Nr), endpoint=True)
        R = bm.recombine(P.astype(np.int64).sum(axis=0)[:, :M, :N], e + 1, f + 1, 4)
        C = [host(c) for c in ddg.qd_recombine_tc(M, N, dev(P), dev(e), dev(f))]
        for p in range(4):
            assert np.array_equal(C[p].view(np.int64), R[p].view(np.int64)), (splits, p)
    assert ddg.wait_timeouts() == 0
