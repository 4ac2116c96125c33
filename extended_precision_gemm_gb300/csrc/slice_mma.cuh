// slice_mma.cuh -- the inner product and the tile epilogue of the FP64
// slice-pair GEMM, shared by the kernel that reads part planes and the one
// that forms its parts from hi/lo tiles.
//
// "Multiple Double Arithmetic on NVIDIA Tensor Cores", eqs. (1)-(4): part d
// of the product of two part expansions collects the pairs s + t = d; with
// the pairs of index sum >= 8 dropped these are 36 FP64 matrix products
// P_d = sum_{s+t=d} A_s B_t, d = 0..7, exact below 2^53 (eq. (5)).  Steps 4-5
// (the parts added in double-double arithmetic and scaled back) may run in
// the epilogue when one block holds all of k.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "dd_arith.cuh"

namespace ddg {

__device__ __forceinline__ void dmma(double& c0, double& c1, double a, double b) {
    asm("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0,%1}, {%2}, {%3}, {%0,%1};"
        : "+d"(c0), "+d"(c1)
        : "d"(a), "d"(b));
}

// One k-chunk (8 values of k) of all 36 pairs for the warp's 16x16 quadrant
// of the tile: rows mq*16 + {0..15}, columns nq*16 + {0..15}, i.e. m8n8
// blocks mb in {2mq, 2mq+1} and nb in {2nq, 2nq+1}.  acc[d][i][j][2] holds
// index sum d of block (2mq+i, 2nq+j).  Every warp runs the same instruction
// stream.  Within a k4 step the B fragments of all 8 parts are loaded once;
// then for each part s of A the 8-s pairs (s, t) are issued, so consecutive
// updates of one accumulator are at least 4 * (8 - s) >= 4 MMAs apart.
__device__ __forceinline__ void chunk_products(const double* __restrict__ As,
                                               const double* __restrict__ Bs, int lane, int mq,
                                               int nq, double (&acc)[S][2][2][2]) {
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) {
        double b[S][2];
#pragma unroll
        for (int t = 0; t < S; ++t)
#pragma unroll
            for (int j = 0; j < 2; ++j) b[t][j] = Bs[((t * (BK / 4) + q) * TN + (2 * nq + j) * 8) * 4 + lane];
#pragma unroll
        for (int s = 0; s < S; ++s) {
            double a[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) a[i] = As[((s * (BK / 4) + q) * TM + (2 * mq + i) * 8) * 4 + lane];
#pragma unroll
            for (int t = 0; t + s < S; ++t)
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j) dmma(acc[s + t][i][j][0], acc[s + t][i][j][1], a[i], b[t][j]);
        }
    }
}

// Tile order of the 128-thread blocks over the 32 x 32 tiles of P: groups of
// 16 row tiles, column-major inside a group, so that the blocks resident at
// one time share few A and B blocks (L2 reuse).
__device__ __forceinline__ void tile_of(int64_t t, int64_t MT, int64_t NT, int64_t& mt, int64_t& nt) {
    constexpr int64_t TILE_GROUP = 16;
    const int64_t group = t / (TILE_GROUP * NT);
    const int64_t first = group * TILE_GROUP;
    const int64_t rows = min(TILE_GROUP, MT - first);
    const int64_t local = t - group * TILE_GROUP * NT;
    mt = first + local % rows;
    nt = local / rows;
}

// Where a block's accumulators go: the P planes of its k-split (splits x 8 x
// Mp x Np, row-major per plane), or, with all of k in one block, C itself
// through the recombination (exponents e, f; rows >= M / columns >= N are
// padding and not written).
struct TileOut {
    double* P;
    int64_t Mp, Np;
    int64_t p_extent;  // doubles in P (splits x 8 x Mp x Np)
    const int32_t* e;
    const int32_t* f;
    double* C_hi;
    double* C_lo;
    int64_t ldc, M, N;
    bool c_vec;  // C_hi, C_lo 16-byte aligned and ldc even: 16-byte stores
};

inline TileOut recombine_out(int64_t Mp, int64_t Np, const int32_t* e, const int32_t* f, int64_t M, int64_t N,
                             double* C_hi, double* C_lo, int64_t ldc) {
    TileOut o{};
    o.Mp = Mp;
    o.Np = Np;
    o.e = e;
    o.f = f;
    o.C_hi = C_hi;
    o.C_lo = C_lo;
    o.ldc = ldc;
    o.M = M;
    o.N = N;
    o.c_vec = (uintptr_t)C_hi % 16 == 0 && (uintptr_t)C_lo % 16 == 0 && ldc % 2 == 0;
    return o;
}

// Epilogue: for block (mb, nb) of m8n8 the thread holds row mb*8 + lane/4 and
// columns nb*8 + 2(lane%4) + {0, 1} of every index sum d.
template <bool RECOMBINE>
__device__ __forceinline__ void store_tile(const double (&acc)[S][2][2][2], const TileOut& o, int lane, int mq,
                                           int nq, int64_t mt, int64_t nt, int z) {
    if constexpr (!RECOMBINE) {
        const int64_t plane = o.Mp * o.Np;
#pragma unroll
        for (int d = 0; d < S; ++d) {
            double* out = o.P + ((int64_t)z * S + d) * plane;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int64_t row = mt * TM + (2 * mq + i) * 8 + (lane >> 2);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int64_t col = nt * TN + (2 * nq + j) * 8 + 2 * (lane & 3);
                    if (in_bounds(((int64_t)z * S + d) * plane + row * o.Np + col + 1, o.p_extent, kSiteGemmStoreP))
                        *reinterpret_cast<double2*>(out + row * o.Np + col) =
                            make_double2(acc[d][i][j][0], acc[d][i][j][1]);
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int64_t row = mt * TM + (2 * mq + i) * 8 + (lane >> 2);
            if (row >= o.M) continue;
            const int ei = effective_exponent(o.e[row]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int64_t col = nt * TN + (2 * nq + j) * 8 + 2 * (lane & 3);
                double hi[2], lo[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    double part[S];
#pragma unroll
                    for (int d = 0; d < S; ++d) part[d] = acc[d][i][j][c];
                    const int fc = col + c < o.N ? effective_exponent(o.f[col + c]) : 0;
                    recombine_parts(part, ei + fc, hi[c], lo[c]);
                }
                if (!in_bounds(row * o.ldc + min(col + 1, o.N - 1), (o.M - 1) * o.ldc + o.N, kSiteGemmStoreC))
                    continue;
                double* ph = o.C_hi + row * o.ldc + col;
                double* pl = o.C_lo + row * o.ldc + col;
                if (o.c_vec && col + 1 < o.N) {
                    *reinterpret_cast<double2*>(ph) = make_double2(hi[0], hi[1]);
                    *reinterpret_cast<double2*>(pl) = make_double2(lo[0], lo[1]);
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        if (col + c < o.N) { ph[c] = hi[c]; pl[c] = lo[c]; }
                }
            }
        }
    }
}

}  // namespace ddg
