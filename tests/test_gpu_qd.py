"""Quad doubles on the integer pipe (qd_gemm): the 16 int16 parts, the 16
part sums and the four output planes bit for bit against the oracle's model
(oracle.slices_md), and the product within the normwise bound of the exact
oracle (the double-double bound's margin over its unit roundoff, 2^20, on the
quad-double unit 2^-208: 1e-57)."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices_md
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu
QD_GATE = 1e-57

SHAPES = [(40, 33, 29, "uniform_exp20"), (1, 1, 1, "normal"), (33, 7, 70, "normal_rowcol30"),
          (64, 64, 64, "uniform")]


def untile_qd(planes, rows, K):
    Rp = -(-rows // 32) * 32
    Kp = -(-K // 8) * 8
    a = np.asarray(planes).reshape(Rp // 32, Kp // 8, 8, 32, 16)
    return a.transpose(4, 0, 3, 1, 2).reshape(16, Rp, Kp)


def _normwise(C, R, A, B):
    d = sum(C[p] - R[p] for p in range(4))
    return float(np.linalg.norm(d) / (np.linalg.norm(sum(A)) * np.linalg.norm(sum(B))))


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_qd_steps_bit_exact(M, N, K, dist):
    A, B = workloads.make_md(M, N, K, dist, 21, 4)
    tA, tB = [dev(a) for a in A], [dev(b) for b in B]
    pA, e, pB, f = ddg.qd_split(tA, tB)
    C_ref, e_ref, f_ref, DA, DB, P_ref = slices_md.sliced_md_gemm(A, B, 16)
    assert np.array_equal(host(e), e_ref) and np.array_equal(host(f), f_ref)
    gA = untile_qd(host(pA), M, K)
    gB = untile_qd(host(pB), N, K)
    assert np.array_equal(gA[:, :M, :K], DA) and np.array_equal(gB[:, :N, :K], DB.transpose(0, 2, 1))
    assert not gA[:, M:, :].any() and not gA[:, :, K:].any()
    KC = -(-K // 8)
    for splits in sorted({s for s in (1, 2, KC) if 1 <= s <= KC}):
        P = ddg.qd_slice_gemm(M, N, K, pA, pB, splits)
        Ps = host(P).sum(axis=0)
        assert np.array_equal(Ps[:, :M, :N], P_ref)
        C = ddg.qd_recombine(M, N, P, e, f)
        for p in range(4):
            assert np.array_equal(host(C[p]).view(np.int64), C_ref[p].view(np.int64)), p


@pytest.mark.parametrize("M,N,K,dist", SHAPES + [(130, 70, 333, "normal")])
def test_qd_gemm_model_and_exact(M, N, K, dist):
    A, B = workloads.make_md(M, N, K, dist, 22, 4)
    C = [host(c) for c in ddg.qd_gemm([dev(a) for a in A], [dev(b) for b in B])]
    if M * N * K <= 10**6:
        C_ref, *_ = slices_md.sliced_md_gemm(A, B, 16)
        for p in range(4):
            assert np.array_equal(C[p].view(np.int64), C_ref[p].view(np.int64))
    R = oracle.exact_md_gemm(A, B)
    assert _normwise(C, R, A, B) <= QD_GATE
    assert ddg.wait_timeouts() == 0


def test_qd_large_sampled():
    import torch
    M = N = K = 1024
    A, B = workloads.make_md(M, N, K, "uniform_exp20", 23, 4)
    ws = torch.empty(ddg.qd_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    C = ddg.qd_gemm([dev(a) for a in A], [dev(b) for b in B], workspace=ws)
    rows = np.array([0, 17, 511, 1023])
    cols = np.array([0, 3, 500, 1023])
    idx = torch.from_numpy(rows).cuda()
    G = [host(c[idx]) for c in C]
    C_ref, *_ = slices_md.sliced_md_gemm([a[rows] for a in A], [b[:, cols] for b in B], 16)
    for p in range(4):
        assert np.array_equal(G[p][:, cols].view(np.int64), C_ref[p].view(np.int64))
    R = oracle.exact_md_gemm(A, B, rows=rows[:2])
    assert _normwise([g[:2] for g in G], R, [a[rows[:2]] for a in A], B) <= QD_GATE


def test_qd_edges_zero_rows_and_k0():
    import torch
    A, B = workloads.make_md(9, 7, 20, "normal_rowcol30", 24, 4)
    for a in A:
        a[2] = 0.0          # an all-zero row: exponent 0, parts 0, outputs +0
    for b in B:
        b[:, 4] = 0.0
    C = [host(c) for c in ddg.qd_gemm([dev(a) for a in A], [dev(b) for b in B])]
    C_ref, *_ = slices_md.sliced_md_gemm(A, B, 16)
    for p in range(4):
        assert np.array_equal(C[p].view(np.int64), C_ref[p].view(np.int64))
    assert not any(c[2].any() for c in C) and not any(np.signbit(c[2]).any() for c in C)
    z = [torch.zeros((3, 0), dtype=torch.float64, device="cuda") for _ in range(4)]
    zb = [torch.zeros((0, 2), dtype=torch.float64, device="cuda") for _ in range(4)]
    C = ddg.qd_gemm(z, zb)
    assert all(c.shape == (3, 2) and not host(c).any() for c in C)


def test_qd_rejects_k_beyond_bound():
    lib = ddg.load()
    import ctypes
    arr = (ctypes.c_void_p * 4)(1 << 20, 1 << 21, 1 << 22, 1 << 23)
    brr = (ctypes.c_void_p * 4)(1 << 30, 1 << 31, 1 << 32, 1 << 33)
    crr = (ctypes.c_void_p * 4)(1 << 40, 1 << 41, 1 << 42, 1 << 43)
    K = ddg.QD_MAX_K + 1
    assert lib.qd_gemm(2, 2, K, ctypes.cast(arr, ctypes.c_void_p), K, ctypes.cast(brr, ctypes.c_void_p), 2,
                       ctypes.cast(crr, ctypes.c_void_p), 2, None, 0, None) == 2
