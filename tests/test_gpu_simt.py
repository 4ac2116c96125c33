"""The comparator on the GPU: bit for bit against its model, and within the
normwise bound of the exact product."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import simt_dd
from tests.gpu_util import dev, host, normwise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,dist", [(64, 64, 64, "uniform"), (37, 45, 29, "uniform_exp20"), (1, 1, 1, "normal"),
                                        (33, 70, 100, "normal_rowcol30"), (130, 50, 17, "uniform")])
def test_simt_bit_exact_and_accurate(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 8)
    C_hi, C_lo = ddg.dd_gemm_simt(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    M_hi, M_lo = simt_dd.simt_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(host(C_hi).view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), M_lo.view(np.int64))
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(host(C_hi), host(C_lo), R_hi, R_lo, A_hi, A_lo, B_hi, B_lo) <= 1e-26


def test_simt_workload1_sampled():
    import torch
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(1)
    C_hi, C_lo = ddg.dd_gemm_simt(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    rows = np.array([0, 5, 511, 1023])
    G_hi = host(C_hi[torch.from_numpy(rows).cuda()])
    G_lo = host(C_lo[torch.from_numpy(rows).cuda()])
    M_hi, M_lo = simt_dd.simt_dd_gemm(A_hi[rows], A_lo[rows], B_hi, B_lo)
    assert np.array_equal(G_hi.view(np.int64), M_hi.view(np.int64))
    assert np.array_equal(G_lo.view(np.int64), M_lo.view(np.int64))
    R_hi, R_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=rows)
    assert normwise(G_hi, G_lo, R_hi, R_lo, A_hi[rows], A_lo[rows], B_hi, B_lo) <= 1e-26
