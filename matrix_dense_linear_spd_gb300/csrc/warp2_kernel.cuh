// Lane-row Cholesky on whole squares with the rows held as float2 column pairs ("warp...:v2=1"),
// f32 potrf: the method and data path of warp_kernel.cuh (one matrix per P lanes, lane l holds
// rows l, l+P, ...; whole-square slabs filled by cp.async while the previous group is factored;
// the column published through a double-buffered shared-memory slot) with the rank-1 update in
// packed two-lane FP32 FMAs on the column pairs (2kk, 2kk+1) of a row.
//
// The differences from the packed variant of warp_kernel.cuh: (1) the register layout: each
// column pair of a row IS a float2, so the packed FMAs read and write their operands in place
// and a 16-byte column load supplies two ready pairs; (2) the store: whole squares have lda = N
// and item stride N*N, so every store offset inside an item is an immediate and the per-column
// address arithmetic disappears (ncu, f32 n=32: ALU instructions 273 -> 245 per matrix, with
// the look-ahead pivots 22.9 us instead of 24.6 us per call at batch 16384, Upper 26.0 instead
// of 28.8 us).
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "potrf: the tiny tier"): right-
// looking, one column j at a time: the pivot d = A(j,j) reaches the P lanes by one shuffle,
// !(d > 0) fails (first failure wins, info = j+1), L(j,j) = d * rsqrt(d), L(i,j) = A(i,j) *
// rsqrt(d), A(i,k) -= L(i,j) * L(k,j) for j < k <= i.
//
// Slabs: whole squares (stride FSTRIDE, the copy moves only the chunks that meet the triangle) or,
// with CSLAB, compacted triangles (TriSlab, about 56% of the square at n = 32), for geometries
// whose whole-square slabs would hold fewer CTAs per SM than the registers allow.

//
// Look-ahead pivots (LA): the lane that owns row j+1 forms the next pivot,
// A(j+1,j+1) - L(j+1,j)^2, from its own registers right after column j is scaled and shuffles
// it at once, so the pivot chain (shuffle, rsqrt, scale, one FMA, shuffle) no longer waits for
// the column's round trip through shared memory; the trailing update of column j fills that
// chain's latency. The owner lane computes the same fused multiply-add the update applies to
// that entry, and every other operation and its order per entry is that of warp_kernel.cuh's
// packed variant, so the results are bit-identical to it.
#pragma once

#include "bl_types.cuh"
#include "warp_kernel.cuh"

namespace bl {

// Scalar view of entry c of a float2-pair row (c a compile-time index after unrolling).
template <int NP>
__device__ __forceinline__ float &pel(float2 (&row)[NP], int c) {
    return (c & 1) ? row[c >> 1].y : row[c >> 1].x;
}

// Copy one group's contiguous run of whole squares (lda = N, item stride N*N) into compacted
// slabs (TriSlab layout, matrix stride MS). Lane (gg, q) = (lane / (N/E), lane mod (N/E)) owns
// chunk q (rows q*E .. q*E+E-1) of matrix gg and sweeps the columns: source and slab offsets are
// lane-fixed bases plus compile-time constants, and the chunk moves for the columns where it
// meets the referenced triangle (Lower: c < q*E + E; Upper: c >= q*E).
template <bool UPPER, int N, int E, int MS, int G>
__device__ __forceinline__ void compact_copy(float *tri, const float *A0, int lane, int64_t mleft) {
    constexpr int NQ = N / E;
    static_assert(G * NQ == 32, "one lane per (matrix, chunk)");
    using L = TriSlab<N, E>;
    const int gg = lane / NQ, q = lane - gg * NQ;
    if (gg >= mleft) return;
    const float *src = A0 + gg * (N * N) + q * E;
    float *dst = tri + gg * MS + q * E;
#pragma unroll
    for (int t = 0; t < NQ; ++t) {                 // columns E*t .. E*t+E-1 share the test
        if (UPPER ? (q > t) : (q < t)) continue;
#pragma unroll
        for (int c = E * t; c < E * t + E; ++c)
            cp_async_16(dst + (UPPER ? L::up_off(c) : L::lo_off(c) - L::lo_first(c)), src + c * N);
    }
}

// Prefetch group `grp` (whole squares, back to back) into the warp's slab: whole-square slabs
// (stride FSTRIDE) or, with CSLAB, compacted ones (stride MSTRIDE).
template <int P, int R, bool CSLAB>
__device__ __forceinline__ void warp2_prefetch(const BatchArgs &args, float *tri, int64_t grp, int lane) {
    using C = WarpCfg<float, P, R>;
    if constexpr (CSLAB) {
        const float *A0 = static_cast<const float *>(args.A) + grp * C::G * static_cast<int64_t>(C::N * C::N);
        const int64_t mleft = args.batch - grp * C::G;
        if (args.upper) compact_copy<true, C::N, C::E, C::MSTRIDE, C::G>(tri, A0, lane, mleft);
        else compact_copy<false, C::N, C::E, C::MSTRIDE, C::G>(tri, A0, lane, mleft);
        cp_async_commit();
    } else {
        warp_prefetch<float, P, R, true>(args, tri, grp, lane, true);
    }
}

// SOLVE (posv, first pass): up to RHS right-hand sides per item ride along as in the lane-row
// solve kernel: the forward substitution inside the column loop (y_j = b_j / L(j,j) published
// next to the column, rows below subtract L(i,j) * y_j), the backward sweep after the factor
// through a staging slab (the transpose of each block of P rows), the same operations in the
// same order as warp_kernel.cuh's whole-square solve kernel.
template <int P, int R, int MINB, bool LA, bool SOLVE = false, bool CSLAB = false>
__global__ void __launch_bounds__(128, MINB) warp2_kernel(const BatchArgs args) {
    using C = WarpCfg<float, P, R>;
    using L = TriSlab<C::N, C::E>;
    constexpr int N = C::N, G = C::G, E = C::E, CB = C::CB, CBX = C::CBX, LDU = C::LDU;
    constexpr int NP = N / 2, RHS = C::RHS, RB = C::RB;
    constexpr int SLAB = CSLAB ? C::MSTRIDE : C::FSTRIDE;          // per-matrix slab stride
    constexpr size_t SHIFT = CSLAB ? 0 : C::full_shift;             // where the other areas start
    static_assert(N % 4 == 0 && P % 2 == 0, "column pairs and 16-byte column loads");
    extern __shared__ __align__(16) unsigned char smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane / P;
    const int l_in = lane - g * P;
    const int slot = warp * G + g;
    const bool upper = args.upper != 0;
    float *tri = reinterpret_cast<float *>(smem) + warp * G * SLAB;
    float *colbuf = reinterpret_cast<float *>(smem + C::off_col + SHIFT) + slot * C::COLS;
    float *stage = reinterpret_cast<float *>(smem + C::off_stage + SHIFT) + slot * P * LDU;
    const int nrhs = SOLVE ? min(args.nrhs, RHS) : 0;
    float *rsb = SOLVE ? reinterpret_cast<float *>(smem + C::off_rs + SHIFT) + slot * N : nullptr;
    float *xsb = SOLVE ? reinterpret_cast<float *>(smem + C::off_x + SHIFT) + slot * 2 * RB : nullptr;

    const int64_t ngroups = (args.batch + G - 1) / G;
    const int64_t gstep = static_cast<int64_t>(gridDim.x) * C::WARPS;
    int64_t grp = static_cast<int64_t>(blockIdx.x) * C::WARPS + warp;
    if (grp < ngroups) warp2_prefetch<P, R, CSLAB>(args, tri, grp, lane);

    for (; grp < ngroups; grp += gstep) {
        int l = l_in;
        asm volatile("" : "+r"(l));
        const int64_t mat = grp * G + g;
        const bool live = mat < args.batch;

        // ---------------------------------------------------------- pick from the slab
        float2 a[R][NP];
        cp_async_wait_all();
        __syncwarp();
        const float *my = tri + g * SLAB;
        if (!upper) {
#pragma unroll
            for (int c = 0; c < N; ++c)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (P * r + P - 1 < c) continue;          // block r has no row >= c
                    pel(a[r], c) = CSLAB ? my[L::lo_off(c) - L::lo_first(c) + l + P * r]
                                         : my[c * C::NS_L + l + P * r];
                }
        } else {
            // row i of S is column i of A: 16 bytes (two pairs) at a time; in a compacted slab
            // the reads past column i's kept rows land in the next column (entries right of the
            // diagonal of S, never read into the factor) and stay inside the matrix's slab
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 *rowp = reinterpret_cast<const float4 *>(
                    my + (CSLAB ? upper_slab_offset(l + P * r, E) : (l + P * r) * C::NS));
#pragma unroll
                for (int c4 = 0; c4 < (P * r + P) / 4; ++c4) {
                    const float4 v = rowp[c4];
                    a[r][2 * c4] = make_float2(v.x, v.y);
                    a[r][2 * c4 + 1] = make_float2(v.z, v.w);
                }
            }
        }
        __syncwarp();
        if (grp + gstep < ngroups) warp2_prefetch<P, R, CSLAB>(args, tri, grp + gstep, lane);

        // right-hand sides: b[r][c] = B(l + P*r, c)
        float b[SOLVE ? R : 1][SOLVE ? RHS : 1];
        float *Bm = SOLVE ? static_cast<float *>(args.B) + (live ? mat * args.stride_b : 0) : nullptr;
        if (SOLVE) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < RHS; ++c)
                    b[r][c] = (live && c < nrhs) ? Bm[static_cast<int64_t>(c) * args.ldb + l + P * r] : 0.f;
        }

        // ---------------------------------------------------------- factor (+ forward solve)
        unsigned failed = 0;
        float dla = LA ? __shfl_sync(0xffffffffu, a[0][0].x, g * P) : 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            asm volatile("" ::: "memory");                   // keeps the columns in order (registers)
            const int rj = j / P, lj = j - rj * P;
            const float d = LA ? dla : __shfl_sync(0xffffffffu, pel(a[rj], j), g * P + lj);
            const bool ok = d > 0.f;
            const float rs = ok ? rsqrtf(d) : 0.f;
            failed |= ok ? 0u : (1u << j);
            float *col = colbuf + (j & 1) * CBX;
            float2 m2[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < rj) continue;
                const float v = pel(a[r], j) * rs;
                pel(a[r], j) = v;
                col[l + P * r] = v;
                m2[r] = make_float2(-v, -v);
            }
            if (LA && j + 1 < N) {
                const int rj1 = (j + 1) / P, lj1 = (j + 1) - rj1 * P;
                const float t = fmaf(-pel(a[rj1], j), pel(a[rj1], j), pel(a[rj1], j + 1));
                dla = __shfl_sync(0xffffffffu, t, g * P + lj1);
            }
            if (SOLVE && l == lj) {
                // forward substitution, axpy form: y_j = b_j / L(j,j), published next to the column
#pragma unroll
                for (int c = 0; c < RHS; ++c) {
                    b[rj][c] = b[rj][c] * rs;
                    col[CB + c] = b[rj][c];
                }
                rsb[j] = rs;
            }
            __syncwarp();
            if (SOLVE) {
#pragma unroll
                for (int q = 0; q < RB / E; ++q) {
                    const float4 yv = reinterpret_cast<const float4 *>(col + CB)[q];
                    const float ys[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int c = q * E + e;
                        if (c >= RHS) continue;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (P * r + P - 1 <= j) continue;      // no row > j in block r
                            if (l + P * r > j) b[r][c] = fmaf(-pel(a[r], j), ys[e], b[r][c]);
                        }
                    }
                }
            }
            // rank-1 update of the trailing entries k > j, one packed FMA per column pair
#pragma unroll
            for (int q = (j + 1) / 4; q < CB / 4; ++q) {
                const float4 ck = reinterpret_cast<const float4 *>(col)[q];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kk = 2 * q + e;                 // the pair (2kk, 2kk+1)
                    const int k = 2 * kk;
                    if (k + 1 <= j) continue;
                    const float2 cv = e ? make_float2(ck.z, ck.w) : make_float2(ck.x, ck.y);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (P * r + P - 1 < k) continue;      // no row >= k in block r
                        if (k <= j) a[r][kk].y = fmaf(m2[r].x, cv.y, a[r][kk].y);   // only k+1 trails
                        else a[r][kk] = __ffma2_rn(m2[r], cv, a[r][kk]);
                    }
                }
            }
        }
        const int info = failed ? __ffs(failed) : 0;

        // ---------------------------------------------------------- backward solve
        if (SOLVE) {
            // L^T x = y, one block of P rows at a time from the bottom: the block's rows of L are
            // transposed through the staging slab, then x_i is broadcast and rows r < i subtract
            // L(i,r) x_i
#pragma unroll
            for (int rb = R - 1; rb >= 0; --rb) {
                __syncwarp();
                {
                    const int i = P * rb + l;
#pragma unroll
                    for (int k = 0; k < P * rb + P; ++k)
                        if (k < i) stage[l * LDU + k] = pel(a[rb], k);
                }
                __syncwarp();
                for (int ii = P - 1; ii >= 0; --ii) {
                    const int i = P * rb + ii;
                    float *xs = xsb + (i & 1) * RB;
                    if (l == ii) {
                        const float ri = rsb[i];
#pragma unroll
                        for (int c = 0; c < RHS; ++c) {
                            b[rb][c] = b[rb][c] * ri;
                            xs[c] = b[rb][c];
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r <= rb; ++r) {
                        const int rr = l + P * r;
                        if (rr < i) {
                            const float lir = stage[ii * LDU + rr];
#pragma unroll
                            for (int c = 0; c < RHS; ++c) b[r][c] = fmaf(-lir, xs[c], b[r][c]);
                        }
                    }
                }
            }
            __syncwarp();
            if (info == 0 && live) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int c = 0; c < RHS; ++c)
                        if (c < nrhs) Bm[static_cast<int64_t>(c) * args.ldb + l + P * r] = b[r][c];
            }
        }

        // ---------------------------------------------------------- store
        asm volatile("" : "+r"(l));
        // whole squares: lda = N and the item stride is N*N, so every store offset inside the
        // item is an immediate (no address arithmetic per column)
        float *A = static_cast<float *>(args.A) + (live ? mat * static_cast<int64_t>(N * N) : 0);
        if (!upper) {
            if (live) {
                float *Al = A + l;
#pragma unroll
                for (int c = 0; c < N; ++c) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (P * r + P - 1 < c) continue;
                        if (P * r >= c || l + P * r >= c) Al[c * N + P * r] = pel(a[r], c);
                    }
                }
            }
        } else {
            // U(c,i) = L(i,c): column i of U is row i of L; transpose through the staging slab,
            // one block of P rows (= P columns of U) at a time; lanes write consecutive rows of a
            // column of U, 32-bit coalesced stores (per-lane 16-byte pieces of a column of U,
            // 32 lines per store instruction, measured slower: f32 n=32 Upper 28.9 us against 26.0)
#pragma unroll
            for (int cb = 0; cb < R; ++cb) {
                const int c0 = P * cb;
                __syncwarp();
                const int i = c0 + l;
#pragma unroll
                for (int c = 0; c < P * cb + P; ++c)
                    if (c <= i) stage[l * LDU + c] = pel(a[cb], c);
                __syncwarp();
                if (live) {
                    float *Al = A + l;
#pragma unroll
                    for (int ii = 0; ii < P; ++ii) {
                        const int colx = c0 + ii;
#pragma unroll
                        for (int t = 0; t <= cb; ++t) {
                            const int r = l + P * t;
                            if (r <= colx) Al[colx * N + P * t] = stage[ii * LDU + r];
                        }
                    }
                }
            }
        }
        if (live && l == 0) args.info[mat] = info;
    }
    cp_async_wait_all();
}

}  // namespace bl
