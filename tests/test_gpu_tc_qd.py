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
