"""The two ways the product shards, on the CUDA path through the C ABI.

* k-split: every slab of the inner dimension takes its raw exponents
  (dd_exponents), the slabs agree on the elementwise maximum (on several
  devices an all-reduce MAX; here torch.maximum), split against it
  (dd_split_with_exponents / dd_split_bf16_with_exponents), form their own
  slice-pair sums, and the sums of all slabs go to one recombination as
  k-splits.  Every partial sum is an integer, so the result must be the
  unsplit product bit for bit, and equal to the oracle's model of the method.
* 2-D output partition: a row of A and a column of B carry their own
  exponents, so a block of rows of A times a block of columns of B gives
  exactly that block of the full product.
"""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import workloads
from oracle import slices, slices_bf16
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _bits(x):
    return np.ascontiguousarray(x).view(np.int64)


def _raw_exponents_ref(X_hi, axis):
    """Oracle exponents with the all-zero sentinel DDGEMM_EXP_NONE."""
    e = slices.row_exponents(X_hi) if axis == 1 else slices.col_exponents(X_hi)
    zero = ~np.any(X_hi != 0, axis=axis)
    return np.where(zero, ddg.EXP_NONE, e)


def _slab_inputs(M, N, K, dist, seed, cut):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, seed)
    # row 3 of A lives after the first cut only, with a negative exponent;
    # column 2 of B before it only: the maximum over slabs must skip an empty
    # slab's sentinel rather than take 0 from it
    A_hi[3, :cut] = 0.0
    A_lo[3, :cut] = 0.0
    A_hi[3] *= 2.0**-9
    A_lo[3] *= 2.0**-9
    B_hi[cut:, 2] = 0.0
    B_lo[cut:, 2] = 0.0
    B_hi[:, 2] *= 2.0**-17
    B_lo[:, 2] *= 2.0**-17
    A_hi[5] = A_lo[5] = 0.0        # zero in every slab
    return A_hi, A_lo, B_hi, B_lo


@pytest.mark.parametrize("M,N,K,dist,cuts", [
    (70, 45, 300, "normal_rowcol30", [100]),
    (33, 64, 1000, "uniform_exp20", [13, 500, 777]),
    (9, 11, 70, "normal", [35]),
])
def test_exponents_raw(M, N, K, dist, cuts):
    A_hi, A_lo, B_hi, B_lo = _slab_inputs(M, N, K, dist, 31, cuts[0])
    bounds = [0, *cuts, K]
    for k0, k1 in zip(bounds[:-1], bounds[1:]):
        e, f = ddg.exponents(dev(A_hi[:, k0:k1]), dev(B_hi[k0:k1]))
        assert np.array_equal(host(e), _raw_exponents_ref(A_hi[:, k0:k1], 1))
        assert np.array_equal(host(f), _raw_exponents_ref(B_hi[k0:k1], 0))
    # an empty slab: every exponent is the sentinel
    e, f = ddg.exponents(dev(np.zeros((M, 0))), dev(np.zeros((0, N))))
    assert (host(e) == ddg.EXP_NONE).all() and (host(f) == ddg.EXP_NONE).all()


@pytest.mark.parametrize("M,N,K,dist,cuts", [
    (70, 45, 300, "normal_rowcol30", [100]),
    (33, 64, 1000, "uniform_exp20", [13, 500, 777]),
    (9, 11, 70, "normal", [35]),
])
def test_k_slabs_fp64_equal_unsplit(M, N, K, dist, cuts):
    import torch
    A_hi, A_lo, B_hi, B_lo = _slab_inputs(M, N, K, dist, 32, cuts[0])
    bounds = [0, *cuts, K]
    slabs = [(k0, k1) for k0, k1 in zip(bounds[:-1], bounds[1:])]
    ts = [(dev(A_hi[:, a:b]), dev(A_lo[:, a:b]), dev(B_hi[a:b]), dev(B_lo[a:b])) for a, b in slabs]
    ef = [ddg.exponents(t[0], t[2]) for t in ts]
    e = ef[0][0].clone()
    f = ef[0][1].clone()
    for e_s, f_s in ef[1:]:  # the all-reduce MAX
        e = torch.maximum(e, e_s)
        f = torch.maximum(f, f_s)
    Ps = []
    for (a, b), t in zip(slabs, ts):
        pA, pB = ddg.split_with_exponents(*t, e, f)
        splits = ddg.layout(M, N, b - a)[3]
        Ps.append(ddg.slice_gemm(M, N, b - a, pA, pB, splits))
    P = torch.cat(Ps, dim=0)  # the slabs' sums side by side as k-splits
    C_hi, C_lo = ddg.recombine(M, N, P, e, f, splits=P.shape[0])
    U_hi, U_lo = ddg.dd_gemm(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    assert np.array_equal(_bits(host(C_hi)), _bits(host(U_hi)))
    assert np.array_equal(_bits(host(C_lo)), _bits(host(U_lo)))
    R_hi, R_lo, *_ = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(_bits(host(C_hi)), _bits(R_hi))
    assert np.array_equal(_bits(host(C_lo)), _bits(R_lo))
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("M,N,K,dist,cuts", [
    (70, 45, 300, "normal_rowcol30", [100]),
    (300, 260, 9000, "uniform_exp20", [4000]),
    (9, 11, 70, "normal", [35]),
])
def test_k_slabs_bf16_equal_unsplit(M, N, K, dist, cuts):
    import torch
    A_hi, A_lo, B_hi, B_lo = _slab_inputs(M, N, K, dist, 33, cuts[0])
    bounds = [0, *cuts, K]
    slabs = [(k0, k1) for k0, k1 in zip(bounds[:-1], bounds[1:])]
    ts = [(dev(A_hi[:, a:b]), dev(A_lo[:, a:b]), dev(B_hi[a:b]), dev(B_lo[a:b])) for a, b in slabs]
    ef = [ddg.exponents(t[0], t[2]) for t in ts]
    e = torch.maximum(ef[0][0], ef[1][0])
    f = torch.maximum(ef[0][1], ef[1][1])
    for e_s, f_s in ef[2:]:
        e = torch.maximum(e, e_s)
        f = torch.maximum(f, f_s)
    Ps = []
    for (a, b), t in zip(slabs, ts):
        pA, pB = ddg.split_bf16_with_exponents(*t, e, f)
        splits = ddg.tc_layout(M, N, b - a)[3]
        Ps.append(ddg.slice_gemm_tc(M, N, b - a, pA, pB, splits))
    P = torch.cat(Ps, dim=0)
    C_hi, C_lo = ddg.recombine_tc(M, N, P, e, f, splits=P.shape[0])
    U_hi, U_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    assert np.array_equal(_bits(host(C_hi)), _bits(host(U_hi)))
    assert np.array_equal(_bits(host(C_lo)), _bits(host(U_lo)))
    if K <= 1000:
        R_hi, R_lo, *_ = slices_bf16.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
        assert np.array_equal(_bits(host(C_hi)), _bits(R_hi))
        assert np.array_equal(_bits(host(C_lo)), _bits(R_lo))
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("gemm", ["dd_gemm", "dd_gemm_tc"])
def test_output_blocks_equal_full_product(gemm):
    M, N, K = 300, 290, 200
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal_rowcol30", 34)
    tA_hi, tA_lo, tB_hi, tB_lo = dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo)
    fn = getattr(ddg, gemm)
    F_hi, F_lo = fn(tA_hi, tA_lo, tB_hi, tB_lo)
    F_hi, F_lo = host(F_hi), host(F_lo)
    # a 2 x 3 grid of uneven blocks, B's column blocks as strided views
    for r0, r1 in [(0, 37), (37, 300)]:
        for c0, c1 in [(0, 101), (101, 257), (257, 290)]:
            G_hi, G_lo = fn(tA_hi[r0:r1], tA_lo[r0:r1], tB_hi[:, c0:c1], tB_lo[:, c0:c1])
            assert np.array_equal(_bits(host(G_hi)), _bits(F_hi[r0:r1, c0:c1]))
            assert np.array_equal(_bits(host(G_lo)), _bits(F_lo[r0:r1, c0:c1]))


def _window(X, offset):
    """X as a column window of a wider device matrix starting `offset`
    elements in (offset 1: rows off the 16-byte grid, odd leading dimension)."""
    import torch
    r, c = X.shape
    big = torch.full((r, c + offset + 1), 7.0, dtype=torch.float64, device="cuda")
    big[:, offset:offset + c] = torch.from_numpy(np.ascontiguousarray(X)).cuda()
    return big[:, offset:offset + c]


@pytest.mark.parametrize("M,N,K", [(3, 65, 4095), (4, 64, 4097), (5, 130, 8200), (6, 33, 63), (7, 129, 65),
                                   (2, 3, 1)])
@pytest.mark.parametrize("offset", [0, 1])
def test_exponents_across_work_items(M, N, K, offset):
    """The exponent pass reduces a row of A in segments of 4096 k and a column
    of B in segments of 64 k (maxima combined across blocks), two columns per
    lane when B is 16-byte aligned with an even leading dimension, one
    otherwise.  Each row's / column's largest element sits at a segment edge
    (first or last k of a segment, or K - 1); one row and one column are all
    zero (the sentinel); one row holds only subnormals."""
    rng = np.random.default_rng(1000 * M + K + offset)
    A_hi = rng.uniform(-1, 1, (M, K)) * 2.0 ** rng.integers(-40, -20, (M, K)).astype(np.float64)
    B_hi = rng.uniform(-1, 1, (K, N)) * 2.0 ** rng.integers(-40, -20, (K, N)).astype(np.float64)
    edges_a = sorted({0, min(4095, K - 1), min(4096, K - 1), K - 1})
    edges_b = sorted({0, min(63, K - 1), min(64, K - 1), K - 1})
    for i in range(M):
        A_hi[i, edges_a[i % len(edges_a)]] = (-1) ** i * 2.0 ** (i % 5) * 1.5
    for j in range(N):
        B_hi[edges_b[j % len(edges_b)], j] = (-1) ** j * 2.0 ** (j % 7) * 1.25
    A_hi[M - 1] = 0.0
    B_hi[:, N - 1] = 0.0
    if M > 2:
        A_hi[1] = rng.uniform(-1, 1, K) * 2.0**-1060  # subnormal row
    e, f = ddg.exponents(_window(A_hi, offset), _window(B_hi, offset))
    assert np.array_equal(host(e), _raw_exponents_ref(A_hi, 1))
    assert np.array_equal(host(f), _raw_exponents_ref(B_hi, 0))
    assert ddg.wait_timeouts() == 0
