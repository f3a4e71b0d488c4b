// Lane-row Cholesky family ("warp"): one matrix per P lanes of a warp (G = 32/P matrices per
// warp), each lane holding R rows in registers, for n <= P*R <= 32.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "potrf: the tiny tier": lanes own
// rows in registers, cross-lane values go by shuffles, no barriers beyond the warp): right-looking
// Cholesky one column j at a time -- pivot d = A(j,j) from its owner lane by one shuffle, fail if
// !(d > 0) (first failure wins, info = j+1), L(j,j) = sqrt(d), L(i,j) = A(i,j)*rsqrt(d),
// then A(i,k) -= L(i,j)*conj(L(k,j)) for j < k <= i.
//
// GB300 layout: lane l of a partition owns rows i = l + P*rho (rho < R), cyclic, so every lane
// keeps trailing work as the matrix shrinks; with R > 1 one warp instruction advances G
// matrices. The column L(:,j) is published once per step into a double-buffered per-partition
// slot in shared memory and read back as 16-byte broadcast loads (one LDS.128 serves four f32
// entries for all lanes), which costs far fewer instructions than one shuffle per entry.
// Lower loads/stores are coalesced per column directly from global memory; Upper reads
// S(i,c) = conj(A(c,i)) through a per-partition staging slab (P columns at a time), so global
// accesses stay coalesced there too.
//
// posv / potrs (same page, "The fused posv tier" and "posv: the backward solve costs a
// transpose"): up to RHS right-hand sides per pass live in registers next to the rows. The
// forward solve L*y = b runs inside the column loop (once column j is scaled, y_j = b_j/L(j,j)
// is broadcast and rows below subtract L(i,j)*y_j). The backward solve L^H*x = y needs row i of
// L, which only its owner lane holds: each block of P rows is written once into the staging
// slab (the transpose through shared memory) and the sweep reads conj(L(i,r)) from there.
// The solve-capable instantiation is separate, so the factor-only kernel keeps its registers.
#pragma once

#include "bl_types.cuh"

namespace bl {

template <typename T, int P, int R>
struct WarpCfg {
    static constexpr int RHS = 8;                    // right-hand sides per solve pass
    static constexpr int N = P * R;
    static constexpr int G = 32 / P;                 // matrices per warp
    static constexpr int WARPS = 4;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int PER_CTA = G * WARPS;
    static constexpr int E = 16 / sizeof(T) > 0 ? 16 / sizeof(T) : 1;  // elements per 16 bytes
    static constexpr int CB = (N + E - 1) / E * E;  // column-buffer length (16-byte multiple)
    static constexpr int RB = (RHS + E - 1) / E * E; // broadcast slots for y_j (16-byte multiple)
    static constexpr int CBX = CB + RB;
    static constexpr int LDU = ((N + 1) % 2) ? N + 1 : N + 2;  // staging leading dim (odd)
    static constexpr int SLOTS = G * WARPS;
    static constexpr size_t col_bytes = sizeof(T) * 2 * CBX * SLOTS;
    static constexpr size_t stage_bytes = sizeof(T) * P * LDU * SLOTS;
    static constexpr size_t off_stage = (col_bytes + 15) / 16 * 16;
    static constexpr size_t off_rs = off_stage + (stage_bytes + 15) / 16 * 16;
    static constexpr size_t rs_bytes = sizeof(real_t<T>) * N * SLOTS;
    static constexpr size_t off_x = off_rs + (rs_bytes + 15) / 16 * 16;
    static constexpr size_t x_bytes = sizeof(T) * 2 * RB * SLOTS;
    static constexpr size_t smem_potrf = off_stage + stage_bytes;
    static constexpr size_t smem_solve = off_x + x_bytes;
};

template <typename T>
struct alignas(16) Vec16 {
    T v[16 / sizeof(T)];
};

template <typename T, int P, int R, bool SOLVE>
__global__ void __launch_bounds__(128) warp_kernel(const BatchArgs args) {
    using C = WarpCfg<T, P, R>;
    using Rt = real_t<T>;
    constexpr int N = C::N, G = C::G, E = C::E, CB = C::CB, CBX = C::CBX, LDU = C::LDU, RHS = C::RHS;
    constexpr int RB = C::RB;
    extern __shared__ __align__(16) unsigned char smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane / P;
    const int l = lane - g * P;
    const int slot = warp * G + g;
    const int64_t mat = static_cast<int64_t>(blockIdx.x) * C::PER_CTA + slot;
    const bool live = mat < args.batch;
    const int n = args.n;
    const bool upper = args.upper != 0;
    const int64_t lda = args.lda;
    T *A = static_cast<T *>(args.A) + (live ? mat * args.stride_a : 0);
    T *colbuf = reinterpret_cast<T *>(smem) + slot * 2 * CBX;
    T *stage = reinterpret_cast<T *>(smem + C::off_stage) + slot * P * LDU;
    const int mode = SOLVE ? args.mode : MODE_POTRF;
    const bool factor = mode != MODE_POTRS;
    const int nrhs = SOLVE ? min(args.nrhs, RHS) : 0;
    T *B = SOLVE ? static_cast<T *>(args.B) + (live ? mat * args.stride_b : 0) : nullptr;
    Rt *rsb = SOLVE ? reinterpret_cast<Rt *>(smem + C::off_rs) + slot * N : nullptr;
    T *xsb = SOLVE ? reinterpret_cast<T *>(smem + C::off_x) + slot * 2 * RB : nullptr;
    // right-hand sides: b[r][c] = B(l + P*r, c)
    T b[SOLVE ? R : 1][SOLVE ? RHS : 1];
    if (SOLVE) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < RHS; ++c) {
                const int i = l + P * r;
                b[r][c] = (live && c < nrhs && i < n) ? B[static_cast<int64_t>(c) * args.ldb + i] : zero<T>();
            }
    }

    T a[R][N];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < N; ++k) a[r][k] = zero<T>();

    // ------------------------------------------------------------------ load
    if (!upper) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
            if (c >= n) break;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (P * r + P - 1 < c) continue;          // block r has no row >= c
                const int i = l + P * r;
                if (live && i < n && i >= c) a[r][c] = A[static_cast<int64_t>(c) * lda + i];
            }
        }
    } else {
#pragma unroll
        for (int cb = 0; cb < R; ++cb) {
            const int c0 = P * cb;
            if (c0 >= n) break;
            // columns c0..c0+P-1 of A are rows c0..c0+P-1 of S; stage their upper parts
            if (live)
                for (int ii = 0; ii < P; ++ii) {
                    const int col = c0 + ii;
                    if (col >= n) break;
                    for (int r = l; r <= col; r += P) stage[ii * LDU + r] = A[static_cast<int64_t>(col) * lda + r];
                }
            __syncwarp();
            const int i = c0 + l;
#pragma unroll
            for (int c = 0; c < P * cb + P; ++c)
                if (c <= i && i < n) a[cb][c] = conj(stage[l * LDU + c]);
            __syncwarp();
        }
    }

    // ------------------------------------------------------------------ factor
    int info = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (j >= n) break;
        const int rj = j / P, lj = j - rj * P;
        const Rt d = __shfl_sync(0xffffffffu, re(a[rj][j]), g * P + lj);
        T *col = colbuf + (j & 1) * CBX;
        Rt rs;
        if (factor) {
            const bool ok = d > Rt(0);
            rs = ok ? rsqrt_of(d) : Rt(0);
            const Rt ljj = ok ? d * rs : d;
            if (!ok && info == 0) info = j + 1;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < rj) continue;
                T v = a[r][j];
                if (r == rj) v = (l == lj) ? from_real<T>(ljj) : (l > lj ? scale(v, rs) : v);
                else v = scale(v, rs);
                a[r][j] = v;
                col[l + P * r] = v;
            }
        } else {
            rs = Rt(1) / d;                                  // the factor is given: 1 / L(j,j)
        }
        if (SOLVE) {
            // forward substitution, axpy form: y_j = b_j / L(j,j), then b_i -= L(i,j) y_j (i > j)
            if (l == lj) {
#pragma unroll
                for (int c = 0; c < RHS; ++c) {
                    b[rj][c] = scale(b[rj][c], rs);
                    if (c < nrhs) col[CB + c] = b[rj][c];
                }
                rsb[j] = rs;
            }
        }
        __syncwarp();
        if (SOLVE) {
#pragma unroll
            for (int q = 0; q < RB / E; ++q) {
                if (q * E >= nrhs) break;
                const Vec16<T> yv = reinterpret_cast<const Vec16<T> *>(col + CB)[q];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int c = q * E + e;
                    if (c >= RHS) continue;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (P * r + P - 1 <= j) continue;          // no row > j in block r
                        const int i = l + P * r;
                        if (i > j) sub_mul(b[r][c], a[r][j], yv.v[e]);
                    }
                }
            }
        }
        if (!factor) continue;
        // rank-1 update of the trailing rows/columns k > j, 16 bytes of the column at a time
#pragma unroll
        for (int q = (j + 1) / E; q < CB / E; ++q) {
            if (q * E >= n) break;
            const Vec16<T> ck = reinterpret_cast<const Vec16<T> *>(col)[q];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int k = q * E + e;
                if (k <= j || k >= N) continue;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (P * r + P - 1 < k) continue;       // no row >= k in block r
                    sub_mul_conj(a[r][k], a[r][j], ck.v[e]);
                }
            }
        }
    }

    // ------------------------------------------------------------------ backward solve
    if (SOLVE) {
        // L^H x = y, one block of P rows at a time from the bottom: the block's rows of L are
        // transposed through the staging slab, then x_i is broadcast and rows r < i subtract
        // conj(L(i,r)) x_i.
#pragma unroll
        for (int rb = R - 1; rb >= 0; --rb) {
            if (P * rb >= n) continue;
            __syncwarp();
            {
                const int i = P * rb + l;
#pragma unroll
                for (int k = 0; k < P * rb + P; ++k)
                    if (k < i) stage[l * LDU + k] = a[rb][k];
            }
            __syncwarp();
            for (int ii = P - 1; ii >= 0; --ii) {
                const int i = P * rb + ii;
                if (i >= n) continue;
                T *xs = xsb + (i & 1) * RB;
                if (l == ii) {
                    const Rt ri = rsb[i];
#pragma unroll
                    for (int c = 0; c < RHS; ++c) {
                        b[rb][c] = scale(b[rb][c], ri);
                        if (c < nrhs) xs[c] = b[rb][c];
                    }
                }
                __syncwarp();
#pragma unroll
                for (int r = 0; r <= rb; ++r) {
                    const int rr = l + P * r;
                    if (rr < i) {
                        const T lir = conj(stage[ii * LDU + rr]);
#pragma unroll
                        for (int c = 0; c < RHS; ++c)
                            if (c < nrhs) sub_mul(b[r][c], lir, xs[c]);
                    }
                }
            }
        }
        __syncwarp();
    }

    // ------------------------------------------------------------------ store
    if (SOLVE && !factor) {
        // solve only: the factor is read-only; a pass after a posv pass skips failed items
        const bool solved = args.info == nullptr || !live || args.info[mat] == 0;
        if (live && solved)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < RHS; ++c) {
                    const int i = l + P * r;
                    if (c < nrhs && i < n) B[static_cast<int64_t>(c) * args.ldb + i] = b[r][c];
                }
        return;
    }
    if (SOLVE && info == 0 && live) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < RHS; ++c) {
                const int i = l + P * r;
                if (c < nrhs && i < n) B[static_cast<int64_t>(c) * args.ldb + i] = b[r][c];
            }
    }
    if (!upper) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
            if (c >= n) break;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (P * r + P - 1 < c) continue;
                const int i = l + P * r;
                if (live && i < n && i >= c) A[static_cast<int64_t>(c) * lda + i] = a[r][c];
            }
        }
    } else {
        __syncwarp();
#pragma unroll
        for (int cb = 0; cb < R; ++cb) {
            const int c0 = P * cb;
            if (c0 >= n) break;
            const int i = c0 + l;
#pragma unroll
            for (int c = 0; c < P * cb + P; ++c)
                if (c <= i && i < n) stage[l * LDU + c] = conj(a[cb][c]);
            __syncwarp();
            if (live)
                for (int ii = 0; ii < P; ++ii) {
                    const int colx = c0 + ii;
                    if (colx >= n) break;
                    for (int r = l; r <= colx; r += P) A[static_cast<int64_t>(colx) * lda + r] = stage[ii * LDU + r];
                }
            __syncwarp();
        }
    }
    if (live && l == 0) args.info[mat] = info;
}

}  // namespace bl
