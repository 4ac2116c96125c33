"""The variant with 8-bit parts on the bf16 tensor cores (tcgen05): its parts,
its part sums P_d and its C must equal the oracle's model of that variant
(oracle.slices_bf16) bit for bit, and C must stay within the normwise bound of
the exact product."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import oracle
import workloads
from oracle import slices, slices_bf16 as sb
from tests.gpu_util import dev, host, normwise, special_dd

pytestmark = pytest.mark.gpu

GATE = 1e-26
SHAPES = [
    (128, 256, 64, "uniform"),           # one block of each operand, one k-block
    (37, 45, 29, "uniform_exp20"),       # ragged everywhere
    (1, 1, 1, "normal"),
    (130, 260, 200, "normal_rowcol30"),  # two row blocks, two column blocks, ragged k
    (5, 300, 321, "uniform"),
    (200, 40, 8, "normal"),
]


def bf16_values(bits):
    """bf16 bit patterns (int16 array) -> their values as int64 (exact integers)."""
    b = (np.asarray(bits).astype(np.int64) & 0xFFFF).astype(np.uint32) << 16
    v = b.view(np.float32).astype(np.float64)
    assert np.array_equal(v, np.round(v))
    return v.astype(np.int64)


def unswizzle(planes, Rp, K, block_rows, parts=sb.S):
    """Part blocks (block, s, kb) of block_rows x 64 in the 128-byte swizzled
    layout of include/ddgemm.h -> D[s, row, k] for Rp padded rows."""
    Kp = -(-K // 64) * 64
    KB = Kp // 64
    a = bf16_values(planes).reshape(Rp // block_rows, parts, KB, block_rows, 8, 8)  # [blk][s][kb][r][pchunk][e]
    r = np.arange(block_rows)
    out = np.empty_like(a)
    for kc in range(8):
        out[:, :, :, r, kc, :] = a[:, :, :, r, kc ^ (r % 8), :]
    return out.transpose(1, 0, 3, 2, 4, 5).reshape(parts, Rp, Kp)


def pad(n, m):
    return -(-n // m) * m


def model(A_hi, A_lo, B_hi, B_lo):
    e, f = sb.row_exponents(A_hi), sb.col_exponents(B_hi)
    DA = sb.split_rows(A_hi, A_lo, e)
    DB = sb.split_cols(B_hi, B_lo, f)
    return e, f, DA, DB


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_split_bf16_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 7)
    pA, e, pB, f = ddg.split_bf16(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    e_ref, f_ref, DA_ref, DB_ref = model(A_hi, A_lo, B_hi, B_lo)
    # the exponent arrays hold the 13-bit method's exponents; the parts use + 1
    assert np.array_equal(host(e) + 1, e_ref) and np.array_equal(host(f) + 1, f_ref)
    DA = unswizzle(host(pA), pad(M, ddg.TC_TILE_M), K, ddg.TC_BLOCK_M)
    DB = unswizzle(host(pB), pad(N, ddg.TC_TILE_N), K, ddg.TC_TILE_N)
    assert np.array_equal(DA[:, :M, :K], DA_ref)
    assert np.array_equal(DB[:, :N, :K], DB_ref.transpose(0, 2, 1))
    assert not DA[:, M:, :].any() and not DA[:, :, K:].any()
    assert not DB[:, N:, :].any() and not DB[:, :, K:].any()


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_slice_gemm_tc_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 7)
    pA, _, pB, _ = ddg.split_bf16(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    _, _, DA, DB = model(A_hi, A_lo, B_hi, B_lo)
    P_ref = sb.slice_products(DA, DB)
    KB = -(-K // 64)
    for splits in sorted({s for s in (1, 2, 3, KB) if 1 <= s <= KB}):
        P = host(ddg.slice_gemm_tc(M, N, K, pA, pB, splits)).astype(np.int64)
        assert np.array_equal(P.sum(axis=0)[:, :M, :N], P_ref), splits
        assert not P[:, :, M:, :].any() and not P[:, :, :, N:].any()
    assert ddg.wait_timeouts() == 0


@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_recombine_tc_bit_exact(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 7)
    pA, e, pB, f = ddg.split_bf16(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    sp = ddg.tc_layout(M, N, K)[3]
    P = ddg.slice_gemm_tc(M, N, K, pA, pB, sp)
    C_hi, C_lo = ddg.recombine_tc(M, N, P, e, f)
    Ps = host(P).astype(np.int64).sum(axis=0)[:, :M, :N]
    R_hi, R_lo = sb.recombine(Ps, host(e) + 1, host(f) + 1)
    assert np.array_equal(host(C_hi).view(np.int64), R_hi.view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), R_lo.view(np.int64))



def _digits_of_sum(Z):
    """13 part sums whose exact sum sum_d v_d 256^(12-d) is Z (v_0 = the bits
    above 96, base-256 digits below; all negated for a negative Z)."""
    s, a = (-1, -Z) if Z < 0 else (1, Z)
    v = [(a >> (8 * (12 - d))) & 0xFF for d in range(1, 13)]
    return [s * (a >> 96)] + [s * x for x in v]


def test_recombine_tc_rounding_cases():
    """Crafted part sums of one k-split against the oracle's rounding: ties of
    the leading and the trailing double (to even, either way), carries to the
    next power of two, exact small values, zero, both signs, the size limit of
    the 128-bit path (|v_0| = 2^30) and scales at the ends of the normal range;
    then random int32 part sums with one and two k-splits."""
    crafted = [
        (2**52 + 1) * 2**60 + 2**59,        # tie, odd 53-bit significand: up
        2**52 * 2**60 + 2**59,              # tie, even: down
        (2**52 + 1) * 2**60 + 2**59 + 1,    # just above the tie
        (2**53 + 1) * 2**60 + 2**59,        # above half an ulp
        2**120 + (2**52 + 1) * 8 + 4,       # exact leading double, tie in the trailing one
        2**120 + 2**52 * 8 + 4,
        2**124 - 1,                         # rounds up to 2^124, trailing -1
        12345, 1, 0,
        (2**30 - 1) * 2**96 + 2**95 + 12345,
        2**30 * 2**96 + 2**77 + 3,          # v_0 = 2^30: outside the 128-bit path
        -(2**30) * 2**96 - 2**70 - 1,       # v_0 = -2^30 (inside) ...
        -(2**30 + 1) * 2**96 + 5,           # ... and -2^30 - 1 (outside)
    ]
    crafted += [-z for z in crafted if z]
    rng = np.random.default_rng(21)
    E = [0, -912, -913, 700, 1000, 1010, -1000]  # q = e + f - 110: -1022 and -1023 at f = 0
    M, Nc, Nr = len(E), len(crafted), 200
    N = Nc + Nr
    Mp, Np = pad(M, ddg.TC_TILE_M), pad(N, ddg.TC_TILE_N)
    e = np.array(E, dtype=np.int32)
    f = np.concatenate([np.zeros(Nc), rng.integers(-6, 7, Nr)]).astype(np.int32)
    for splits in (1, 2):
        P = np.zeros((splits, sb.S, Mp, Np), dtype=np.int32)
        for c, Z in enumerate(crafted):
            P[0, :, :M, c] = np.array(_digits_of_sum(Z), dtype=np.int64)[:, None]
        lim = np.iinfo(np.int32)
        P[:, :, :M, Nc:N] = rng.integers(lim.min, lim.max, (splits, sb.S, M, Nr), endpoint=True)
        half = Nc + Nr // 2                 # half of the random columns inside the 128-bit path
        P[:, 0, :M, Nc:half] = rng.integers(-2**30 // splits, 2**30 // splits, (splits, M, half - Nc))
        R_hi, R_lo = sb.recombine(P.astype(np.int64).sum(axis=0)[:, :M, :N], e + 1, f + 1)
        C_hi, C_lo = ddg.recombine_tc(M, N, dev(P), dev(e), dev(f))
        assert np.array_equal(host(C_hi).view(np.int64), R_hi.view(np.int64)), splits
        assert np.array_equal(host(C_lo).view(np.int64), R_lo.view(np.int64)), splits
        # part sums 4 bytes off a 16-byte boundary, C with an odd leading dimension
        flat = dev(np.concatenate([np.zeros(1, np.int32), P.ravel()]))
        Pm = flat[1:].view(P.shape)
        Wh, Wl = dev(np.zeros((M, N + 1))), dev(np.zeros((M, N + 1)))
        ddg.recombine_tc(M, N, Pm, dev(e), dev(f), None, Wh[:, :N], Wl[:, :N])
        assert np.array_equal(host(Wh)[:, :N].view(np.int64), R_hi.view(np.int64)), splits
        assert np.array_equal(host(Wl)[:, :N].view(np.int64), R_lo.view(np.int64)), splits
    assert ddg.wait_timeouts() == 0

@pytest.mark.parametrize("M,N,K,dist", SHAPES)
def test_dd_gemm_tc_matches_model_and_bound(M, N, K, dist):
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 11)
    C_hi, C_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    R = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(host(C_hi).view(np.int64), R[0].view(np.int64))
    assert np.array_equal(host(C_lo).view(np.int64), R[1].view(np.int64))
    X_hi, X_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(host(C_hi), host(C_lo), X_hi, X_lo, A_hi, A_lo, B_hi, B_lo) <= GATE
    assert ddg.wait_timeouts() == 0


def test_dd_gemm_tc_special_values_and_strides():
    rng = np.random.default_rng(17)
    A_hi, A_lo = special_dd(rng, 70, 90)
    B_hi, B_lo = special_dd(rng, 90, 50)
    A_hi[3, :] = A_lo[3, :] = 0.0          # zero row: exponent 0, C row +0
    B_hi[:, 7] = B_lo[:, 7] = 0.0          # zero column
    import torch
    pad = torch.zeros((70, 101), dtype=torch.float64).cuda()
    Ah, Al = pad.clone(), pad.clone()
    Ah[:, :90] = dev(A_hi)
    Al[:, :90] = dev(A_lo)
    Ch = torch.full((70, 64), 7.0, dtype=torch.float64).cuda()
    Cl = torch.full((70, 64), 7.0, dtype=torch.float64).cuda()
    ddg.dd_gemm_tc(Ah[:, :90], Al[:, :90], dev(B_hi), dev(B_lo), Ch[:, :50], Cl[:, :50])
    R = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    C_hi, C_lo = host(Ch), host(Cl)
    assert np.array_equal(C_hi[:, :50].view(np.int64), R[0].view(np.int64))
    assert np.array_equal(C_lo[:, :50].view(np.int64), R[1].view(np.int64))
    assert (C_hi[:, 50:] == 7.0).all() and (C_lo[:, 50:] == 7.0).all()
    assert not np.signbit(C_hi[3, :50]).any() and not C_hi[3, :50].any()
    X = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(C_hi[:, :50], C_lo[:, :50], *X, A_hi, A_lo, B_hi, B_lo) <= GATE


def test_dd_gemm_tc_empty_and_k0():
    import torch
    z = torch.zeros((0, 5), dtype=torch.float64).cuda()
    C_hi, C_lo = ddg.dd_gemm_tc(z, z, torch.zeros((5, 3), dtype=torch.float64).cuda(),
                                torch.zeros((5, 3), dtype=torch.float64).cuda())
    assert C_hi.shape == (0, 3)
    A = torch.zeros((4, 0), dtype=torch.float64).cuda()
    B = torch.zeros((0, 6), dtype=torch.float64).cuda()
    C_hi = torch.full((4, 6), 3.0, dtype=torch.float64).cuda()
    C_lo = torch.full((4, 6), 3.0, dtype=torch.float64).cuda()
    ddg.dd_gemm_tc(A, A, B, B, C_hi, C_lo)
    assert not host(C_hi).any() and not host(C_lo).any()
    assert not np.signbit(host(C_hi)).any()


def test_k_beyond_one_split_is_split_and_exact():
    # K = 9000 > 8192: at least two k-splits, each with exact int32 sums
    M, N, K = 6, 20, 9000
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 23)
    Mp, Np, Kp, sp = ddg.tc_layout(M, N, K)
    assert sp >= 2 and -(-(Kp // 64) // sp) * 64 <= ddg.TC_MAX_K_SPLIT
    pA, e, pB, f = ddg.split_bf16(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    P = host(ddg.slice_gemm_tc(M, N, K, pA, pB, sp)).astype(np.int64).sum(axis=0)[:, :M, :N]
    _, _, DA, DB = model(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(P, sb.slice_products(DA, DB))
    with pytest.raises(ddg.DDGemmError):
        ddg.slice_gemm_tc(M, N, K, pA, pB, 1)      # one split would overflow int32
    C_hi, C_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    X = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert normwise(host(C_hi), host(C_lo), *X, A_hi, A_lo, B_hi, B_lo) <= GATE


def _extreme_element():
    """A double double whose parts (exponent e' = 0) are -127 then twelve times
    -128: every product of two lower parts is 2^14, so a chunk of 1024 of them
    sums to exactly 2^24, the bound of the f32 accumulation."""
    from fractions import Fraction
    X = -(127 * 256**12 + 128 * (256**12 - 1) // 255)
    v = Fraction(X, 2**104)
    hi = float(v)
    lo = float(v - Fraction(hi))
    assert Fraction(hi) + Fraction(lo) == v
    return hi, lo


@pytest.mark.parametrize("K", [512, 1024, 2048])
def test_largest_parts_accumulate_exactly(K):
    # with K = 1024 a chunk of one pair (s, t >= 1) sums 1024 products of
    # 128 x 128: exactly 2^24 in the f32 accumulator
    hi, lo = _extreme_element()
    M, N = 128, 256
    A_hi, A_lo = np.full((M, K), hi), np.full((M, K), lo)
    B_hi, B_lo = np.full((K, N), hi), np.full((K, N), lo)
    assert sb.digits_of(hi, lo, 0) == [-127] + [-128] * 12
    pA, e, pB, f = ddg.split_bf16(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    assert (host(e) == -1).all() and (host(f) == -1).all()
    DA = unswizzle(host(pA), pad(M, ddg.TC_TILE_M), K, ddg.TC_BLOCK_M)
    assert (DA[0, :M] == -127).all() and (DA[1:, :M] == -128).all()
    P = host(ddg.slice_gemm_tc(M, N, K, pA, pB, 1)).astype(np.int64)[0]
    _, _, DAr, DBr = model(A_hi[:2], A_lo[:2], B_hi[:, :2], B_lo[:, :2])
    P_ref = sb.slice_products(DAr, DBr)
    assert P_ref[12, 0, 0] == K * (2 * 127 * 128 + 11 * 128 * 128)
    assert np.array_equal(P[:, :2, :2], P_ref)
    assert np.all(P[:, :M, :N] == P[:, :1, :1])   # every output identical
    C_hi, C_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    X = oracle.exact_dd_gemm(A_hi[:2], A_lo[:2], B_hi[:, :2], B_lo[:, :2])
    assert normwise(host(C_hi)[:2, :2], host(C_lo)[:2, :2], *X, A_hi[:2], A_lo[:2], B_hi[:, :2], B_lo[:, :2]) <= GATE
    assert ddg.wait_timeouts() == 0


def test_rejects_bad_arguments():
    import torch
    A = torch.zeros((4, 4), dtype=torch.float64).cuda()
    with pytest.raises(ddg.DDGemmError):
        ddg.dd_gemm_tc(A, A, A, A, A, A)          # C overlaps A
    lib = ddg.load()
    assert lib.dd_gemm_tc(4, 4, ddg.MAX_K + 1, 1, 1, ddg.MAX_K + 1, 1, 1, 4, 1, 1, 4, None, 0, None) == 2
    assert lib.dd_slice_gemm_tc(4, 4, 64, 16, 16, 0, 16, None) == 1       # splits < 1


def test_dd_gemm_tc_host_matches_device_and_model():
    # host operands and result: copies in, the product, the copy back, with
    # leading dimensions of the host arrays larger than their widths
    M, N, K = 130, 260, 200
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal_rowcol30", 24)
    D_hi, D_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    H_hi = np.zeros((M, N))
    H_lo = np.zeros((M, N))
    ddg.dd_gemm_tc_host(A_hi, A_lo, B_hi, B_lo, H_hi, H_lo)
    assert np.array_equal(H_hi.view(np.int64), host(D_hi).view(np.int64))
    assert np.array_equal(H_lo.view(np.int64), host(D_lo).view(np.int64))
    R_hi, R_lo, *_ = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(H_hi.view(np.int64), R_hi.view(np.int64))
    assert np.array_equal(H_lo.view(np.int64), R_lo.view(np.int64))
    lib = ddg.load()
    wide = np.zeros((M, K + 3))
    widel = np.zeros((M, K + 3))
    wide[:, :K], widel[:, :K] = A_hi, A_lo
    Cw = np.full((M, N + 2), 5.0)
    Cwl = np.full((M, N + 2), 5.0)
    assert lib.dd_gemm_tc_host(M, N, K, wide.ctypes.data, widel.ctypes.data, K + 3, B_hi.ctypes.data,
                               B_lo.ctypes.data, N, Cw.ctypes.data, Cwl.ctypes.data, N + 2, None) == 0
    assert np.array_equal(Cw[:, :N], H_hi) and np.array_equal(Cwl[:, :N], H_lo)
    assert (Cw[:, N:] == 5.0).all() and (Cwl[:, N:] == 5.0).all()
    # the pool that keeps the calls' device memory can be emptied, and the
    # next call refills it
    ddg.pool_trim()
    G_hi = np.zeros((M, N))
    G_lo = np.zeros((M, N))
    ddg.dd_gemm_tc_host(A_hi, A_lo, B_hi, B_lo, G_hi, G_lo)
    ddg.dd_gemm_host(A_hi, A_lo, B_hi, B_lo, np.zeros((M, N)), np.zeros((M, N)))
    assert np.array_equal(G_hi, H_hi) and np.array_equal(G_lo, H_lo)
    ddg.pool_trim()


def test_dd_gemm_tc_host_pipelined_blocks():
    # M >= 1024: A goes up in blocks of rows while earlier blocks compute and
    # finished blocks of C come back (here blocks of 512, 512 and 76 rows);
    # the result must be the one-shot device product's, and the oracle
    # model's, bit for bit, with leading dimensions above the widths
    M, N, K = 1100, 300, 200
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "uniform_exp20", 25)
    D_hi, D_lo = ddg.dd_gemm_tc(dev(A_hi), dev(A_lo), dev(B_hi), dev(B_lo))
    wide, widel = np.zeros((M, K + 5)), np.zeros((M, K + 5))
    wide[:, :K], widel[:, :K] = A_hi, A_lo
    Bw, Bwl = np.zeros((K, N + 3)), np.zeros((K, N + 3))
    Bw[:, :N], Bwl[:, :N] = B_hi, B_lo
    Cw = np.full((M, N + 2), 5.0)
    Cwl = np.full((M, N + 2), 5.0)
    lib = ddg.load()
    for _ in range(2):  # twice: the second call reuses the pool's memory
        assert lib.dd_gemm_tc_host(M, N, K, wide.ctypes.data, widel.ctypes.data, K + 5, Bw.ctypes.data,
                                   Bwl.ctypes.data, N + 3, Cw.ctypes.data, Cwl.ctypes.data, N + 2, None) == 0
        assert np.array_equal(Cw[:, :N].view(np.int64), host(D_hi).view(np.int64))
        assert np.array_equal(Cwl[:, :N].view(np.int64), host(D_lo).view(np.int64))
        assert (Cw[:, N:] == 5.0).all() and (Cwl[:, N:] == 5.0).all()
    R_hi, R_lo, *_ = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
    assert np.array_equal(Cw[:, :N].view(np.int64), R_hi.view(np.int64))
    assert np.array_equal(Cwl[:, :N].view(np.int64), R_lo.view(np.int64))
    assert ddg.wait_timeouts() == 0
