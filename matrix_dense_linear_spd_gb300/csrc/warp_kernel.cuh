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
#pragma once

#include "bl_types.cuh"

namespace bl {

template <typename T, int P, int R>
struct WarpCfg {
    static constexpr int N = P * R;
    static constexpr int G = 32 / P;                 // matrices per warp
    static constexpr int WARPS = 4;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int PER_CTA = G * WARPS;
    static constexpr int E = 16 / sizeof(T) > 0 ? 16 / sizeof(T) : 1;  // elements per 16 bytes
    static constexpr int CB = (N + E - 1) / E * E;  // column-buffer length (16-byte multiple)
    static constexpr int LDU = ((N + 1) % 2) ? N + 1 : N + 2;  // staging leading dim (odd)
    static constexpr size_t col_bytes = sizeof(T) * 2 * CB * G * WARPS;
    static constexpr size_t stage_bytes = sizeof(T) * P * LDU * G * WARPS;
    static constexpr size_t off_stage = (col_bytes + 15) / 16 * 16;
    static constexpr size_t smem_bytes = off_stage + stage_bytes;
};

template <typename T>
struct alignas(16) Vec16 {
    T v[16 / sizeof(T)];
};

template <typename T, int P, int R>
__global__ void __launch_bounds__(128) warp_kernel(const BatchArgs args) {
    using C = WarpCfg<T, P, R>;
    using Rt = real_t<T>;
    constexpr int N = C::N, G = C::G, E = C::E, CB = C::CB, LDU = C::LDU;
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
    T *colbuf = reinterpret_cast<T *>(smem) + slot * 2 * CB;
    T *stage = reinterpret_cast<T *>(smem + C::off_stage) + slot * P * LDU;

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
        const bool ok = d > Rt(0);
        const Rt rs = ok ? rsqrt_of(d) : Rt(0);
        const Rt ljj = ok ? d * rs : d;
        if (!ok && info == 0) info = j + 1;
        T *col = colbuf + (j & 1) * CB;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < rj) continue;
            T v = a[r][j];
            if (r == rj) v = (l == lj) ? from_real<T>(ljj) : (l > lj ? scale(v, rs) : v);
            else v = scale(v, rs);
            a[r][j] = v;
            col[l + P * r] = v;
        }
        __syncwarp();
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

    // ------------------------------------------------------------------ store
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
