"""Exactness of the bf16 variant's f32 tensor-core accumulation at the edge of
its range, with crafted part blocks fed straight into dd_slice_gemm_tc.

The slice GEMM sums the 8-bit part products of 1024 consecutive products per
output ("a chunk": 64 MMAs of K = 16) in f32 in tensor memory, then converts
the chunk exactly into int32 totals.  Each product is at most 2^14, so every
partial sum is an integer of magnitude at most 2^24, which f32 holds; the
argument for exactness also needs the MMA's internal alignment to keep the
units bit when the accumulator is large.  Before the last MMA of a chunk the
accumulator is at most 1008 * 2^14 = 2^24 - 16 * 2^14 in magnitude.  These
cases put it exactly there, at both signs, and let the last MMA mix products
of 2^14 with products of 1 (cancelling or not, the large addend first or
last).  The expected sums come from the oracle's plain int64 products
(oracle.slices_bf16.slice_products) of the same digits.

Within a unit the MMAs run pair by pair (s = 0..d), each pair over the
split's k-blocks in order, so for the index sum d = 0 a chunk is exactly
k in [1024 c, 1024 (c + 1)); for d = 1 with K = 512 one chunk holds the 512
products of pair (0, 1) followed by the 512 of pair (1, 0)."""
import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
from oracle import slices_bf16 as sb

pytestmark = pytest.mark.gpu

NP = sb.S          # 13 parts
EDGE = 1008        # products of 2^14 before the last MMA of a chunk
M, N = 256, 256    # one CTA pair's output block


def bf16_bits(D):
    """Integer parts (|v| <= 256) -> their bf16 bit patterns as int16."""
    v = np.asarray(D, dtype=np.float32)
    assert np.array_equal(v.astype(np.int64), np.asarray(D))
    return (v.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)


def swizzle(D, block_rows):
    """D[s, row, k] (rows and k padded) -> the part blocks of ddgemm.h: block
    (b, s, kb) of block_rows x 64, element (r, k) at byte r * 128 +
    (((k / 8) ^ (r % 8)) * 16) + (k % 8) * 2."""
    parts, Rp, Kp = D.shape
    KB = Kp // 64
    x = D.reshape(parts, Rp // block_rows, block_rows, KB, 8, 8).transpose(1, 0, 3, 2, 4, 5)  # [b][s][kb][r][kc][e]
    a = np.empty_like(x)
    r = np.arange(block_rows)
    for p in range(8):
        a[:, :, :, r, p, :] = x[:, :, :, r, p ^ (r % 8), :]
    return bf16_bits(a.reshape(-1))


def run(DA, DB):
    """P (13 x M x N, int64) of dd_slice_gemm_tc on digit planes DA[s, i, k],
    DB[t, k, j], one k-split."""
    import torch
    K = DA.shape[2]
    A = swizzle(DA, ddg.TC_BLOCK_M)
    B = swizzle(DB.transpose(0, 2, 1), ddg.TC_TILE_N)
    pA = torch.from_numpy(A).cuda()
    pB = torch.from_numpy(B).cuda()
    P = ddg.slice_gemm_tc(M, N, K, pA, pB, 1)
    return P.cpu().numpy().astype(np.int64)[0]


def tail_patterns(rng, n):
    """n patterns of 16 values for the last MMA of a chunk: crafted mixes of
    2^7-sized and unit-sized parts first, then random ones."""
    crafted = [
        [128] * 15 + [1],                      # large addends, a unit last
        [1] * 15 + [128],                      # units, the large addend last
        [128, -128] * 7 + [128, 1],            # cancelling large pairs, odd remainder
        [1, 128, -1, -128] * 4,                # alternating signs and sizes
        [-128] * 8 + [1, -1] * 4,              # eight large of one sign, units
        [127, -127, 1, 0] * 4,
        [0] * 15 + [1],
        [128] * 16,                            # reaches 2^24 exactly with +128 columns
    ]
    vals = np.array([128, -128, 127, -127, 64, 1, -1, 2, -3, 0])
    out = [np.array(c) for c in crafted]
    while len(out) < n:
        out.append(rng.choice(vals, 16))
    return np.stack(out[:n])


@pytest.mark.parametrize("K", [1024, 2048])
def test_chunk_at_the_edge_index_sum_0(K):
    rng = np.random.default_rng(51)
    DA = np.zeros((NP, M, K), dtype=np.int64)
    DB = np.zeros((NP, K, N), dtype=np.int64)
    sign = np.where(np.arange(N) < N // 2, 1, -1)       # +(2^24 - 2^18) and -(2^24 - 2^18)
    for c in range(K // 1024):
        k0 = 1024 * c
        DA[0, :, k0:k0 + EDGE] = 128
        DB[0, k0:k0 + EDGE, :] = 128 * sign[None, :]
        DA[0, :, k0 + EDGE:k0 + 1024] = tail_patterns(rng, M)
        DB[0, k0 + EDGE:k0 + 1024, :] = tail_patterns(rng, N).T
        # the chunk's own sums: within +-2^24, and both edges mixed with
        # large and unit products in the last MMA
        ch = DA[0, :, k0:k0 + 1024] @ DB[0, k0:k0 + 1024, :]
        assert np.abs(ch).max() <= 2**24
        assert ch[:, : N // 2].max() > EDGE * 2**14 and ch[:, N // 2:].min() < -EDGE * 2**14
    P_ref = sb.slice_products(DA, DB)
    P = run(DA, DB)
    assert np.array_equal(P, P_ref)
    assert ddg.wait_timeouts() == 0


def test_chunk_spanning_two_pairs_at_the_edge():
    # index sum 1 with K = 512: one chunk = pair (0, 1) over k < 512 (sum
    # 2^23), then pair (1, 0) whose first 496 products bring the accumulator
    # to 2^24 - 16 2^14 before its last MMA mixes large and unit products
    K = 512
    rng = np.random.default_rng(52)
    DA = np.zeros((NP, M, K), dtype=np.int64)
    DB = np.zeros((NP, K, N), dtype=np.int64)
    sign = np.where(np.arange(N) % 2 == 0, 1, -1)
    DA[0] = 128
    DB[1] = 128 * sign[None, :]
    DA[1, :, :496] = 128
    DB[0, :496, :] = 128 * sign[None, :]
    DA[1, :, 496:] = tail_patterns(rng, M)
    DB[0, 496:, :] = tail_patterns(rng, N).T
    P_ref = sb.slice_products(DA, DB)
    assert np.abs(P_ref[1]).max() <= 2**24
    P = run(DA, DB)
    assert np.array_equal(P, P_ref)
    assert ddg.wait_timeouts() == 0


def test_small_remainders_after_cancellation_in_every_mma():
    # every MMA of a chunk holds +2^14 and -2^14 products that cancel, plus
    # one unit product: the accumulator stays small while each MMA's largest
    # addends are 2^14
    K = 1024
    rng = np.random.default_rng(53)
    DA = np.zeros((NP, M, K), dtype=np.int64)
    DB = np.zeros((NP, K, N), dtype=np.int64)
    base = np.array([128, -128] * 7 + [1, 0])
    for g in range(K // 16):
        DA[0, :, 16 * g:16 * g + 16] = np.roll(base, g % 16)[None, :]
        DB[0, 16 * g:16 * g + 16, :] = 128
        DB[0, 16 * g:16 * g + 16, : N // 2] *= -1
    DB[0, :, ::3] = rng.choice([1, -1, 128], size=(K, len(range(0, N, 3))))
    P_ref = sb.slice_products(DA, DB)
    P = run(DA, DB)
    assert np.array_equal(P, P_ref)
