// Blocked Cholesky family ("blocked"): one CTA per matrix, right-looking over panels of NB
// columns, the matrix updated in place in global memory (L2 holds the active matrices).
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "The blocked driver"): for
// j0 = 0, NB, 2NB, ...
//   1. factor the diagonal block L11 = chol(A11) (in shared memory);
//   2. panel solve L21 = A21 * L11^{-H} (one row per thread, L11 in shared memory);
//   3. trailing update A22 -= L21 * L21^H on the lower triangle only: tiles on or below the
//      diagonal, the diagonal tiles masked, so the other triangle is never written (the page's
//      blocked-driver findings record that an update which skips this masking overwrites the
//      upper triangle).
// A failure at local column c of a panel is reported at global column j0 + c + 1
// ("potrf: correctness findings" item 6), and the item stops there.
// Upper runs on the view S(i,k) = conj(A(k,i)); every global access is mapped so that the
// index that is contiguous in memory varies fastest across threads.
// posv / potrs: after the factor, forward (L*y = b, axpy form) and back (L^H*x = y, axpy form
// on the rows of L) substitution in global memory ("The fused potrs solve").
#pragma once

#include "bl_types.cuh"

namespace bl {

template <typename T>
struct SView {  // the Lower view S of the stored matrix
    T *A;
    int64_t lda;
    bool upper;
    __device__ __forceinline__ T get(int i, int k) const {
        return upper ? conj(A[static_cast<int64_t>(i) * lda + k]) : A[static_cast<int64_t>(k) * lda + i];
    }
    __device__ __forceinline__ void set(int i, int k, T v) const {
        if (upper) A[static_cast<int64_t>(i) * lda + k] = conj(v);
        else A[static_cast<int64_t>(k) * lda + i] = v;
    }
};

template <typename T, int NB>
struct BlkCfg {
    static constexpr int THREADS = 256;
    static constexpr int TB = 64;             // trailing tile edge; 16 x 16 threads x (4 x 4)
    static constexpr int LDD = NB + 1;        // diagonal block leading dimension
    static constexpr int LDP = NB + 1;        // panel-row staging leading dimension
    static constexpr int LDT = TB + 4;        // trailing operand leading dimension
    using R = real_t<T>;
    static constexpr size_t diag_bytes = sizeof(T) * NB * LDD;
    static constexpr size_t rs_bytes = sizeof(R) * NB;
    static constexpr size_t panel_bytes = sizeof(T) * THREADS * LDP;
    static constexpr size_t trail_bytes = sizeof(T) * 2 * NB * LDT;
    static constexpr size_t work_bytes = panel_bytes > trail_bytes ? panel_bytes : trail_bytes;
    static constexpr size_t off_diag = 0;
    static constexpr size_t off_rs = off_diag + diag_bytes;
    static constexpr size_t off_work = ((off_rs + rs_bytes) + 15) / 16 * 16;
    static constexpr size_t smem_bytes = off_work + work_bytes;
};

// 16-byte elements (complex<double>): the 4 x 4 accumulator tile and its operands need more than
// the 64 registers per thread that four 256-thread CTAs per SM leave, so two CTAs per SM.
template <typename T, int NB>
__global__ void __launch_bounds__(256, sizeof(T) >= 16 ? 2 : 4) blocked_kernel(const BatchArgs args) {
    using C = BlkCfg<T, NB>;
    using R = typename C::R;
    constexpr int THREADS = C::THREADS, TB = C::TB, LDD = C::LDD, LDP = C::LDP, LDT = C::LDT;
    extern __shared__ __align__(16) unsigned char smem[];
    T *sD = reinterpret_cast<T *>(smem + C::off_diag);
    R *sRs = reinterpret_cast<R *>(smem + C::off_rs);
    T *sW = reinterpret_cast<T *>(smem + C::off_work);
    __shared__ int s_fail;

    const int tid = threadIdx.x;
    const int64_t mat = blockIdx.x;
    const int n = args.n;
    const int mode = args.mode;
    const bool upper = args.upper != 0;
    const SView<T> S{static_cast<T *>(args.A) + mat * args.stride_a, args.lda, upper};
    // a solve-only pass that follows a posv pass is given info and skips the failed items
    if (tid == 0) s_fail = (mode == MODE_POTRS && args.info != nullptr && args.info[mat] != 0) ? 1 : 0;
    __syncthreads();

    if (mode != MODE_POTRS) {
        for (int j0 = 0; j0 < n; j0 += NB) {
            const int kb = min(NB, n - j0);
            // ---------------------------------------------- 1. diagonal block
            for (int idx = tid; idx < kb * kb; idx += THREADS) {
                // contiguous index fastest: Lower -> row r, Upper -> column c (of S)
                const int a0 = idx % kb, a1 = idx / kb;
                const int r = upper ? a1 : a0, c = upper ? a0 : a1;
                if (r >= c) sD[c * LDD + r] = S.get(j0 + r, j0 + c);
            }
            __syncthreads();
            int fail_col = -1;
            for (int c = 0; c < kb; ++c) {
                const R d = re(sD[c * LDD + c]);
                const bool ok = d > R(0);
                if (!ok) { fail_col = c; break; }            // uniform: every thread read d
                const R rs = rsqrt_of(d);
                __syncthreads();                             // everyone has read the pivot
                if (tid == 0) { sD[c * LDD + c] = from_real<T>(d * rs); sRs[c] = rs; }
                for (int r = c + 1 + tid; r < kb; r += THREADS) sD[c * LDD + r] = scale(sD[c * LDD + r], rs);
                __syncthreads();
                const int m = kb - c - 1;                    // trailing order inside the block
                for (int idx = tid; idx < m * m; idx += THREADS) {
                    const int r = c + 1 + idx % m, k = c + 1 + idx / m;
                    if (r >= k) sub_mul_conj(sD[k * LDD + r], sD[c * LDD + r], sD[c * LDD + k]);
                }
                __syncthreads();
            }
            // store the diagonal block (columns before a failure are final)
            for (int idx = tid; idx < kb * kb; idx += THREADS) {
                const int a0 = idx % kb, a1 = idx / kb;
                const int r = upper ? a1 : a0, c = upper ? a0 : a1;
                if (r >= c) S.set(j0 + r, j0 + c, sD[c * LDD + r]);
            }
            if (fail_col >= 0) {
                if (tid == 0) { args.info[mat] = j0 + fail_col + 1; s_fail = 1; }
                break;
            }
            __syncthreads();
            // ---------------------------------------------- 2. panel solve L21 = A21 L11^{-H}
            const int m0 = j0 + kb;
            for (int rb = m0; rb < n; rb += THREADS) {
                const int nrow = min(THREADS, n - rb);
                for (int idx = tid; idx < nrow * kb; idx += THREADS) {
                    const int a0 = upper ? idx % kb : idx % nrow;
                    const int a1 = upper ? idx / kb : idx / nrow;
                    const int t = upper ? a1 : a0, c = upper ? a0 : a1;
                    sW[t * LDP + c] = S.get(rb + t, j0 + c);
                }
                __syncthreads();
                if (tid < nrow) {
                    T *row = sW + tid * LDP;
                    for (int k = 0; k < kb; ++k) {
                        T x = row[k];
                        for (int m = 0; m < k; ++m) sub_mul_conj(x, row[m], sD[m * LDD + k]);
                        row[k] = scale(x, sRs[k]);
                    }
                }
                __syncthreads();
                for (int idx = tid; idx < nrow * kb; idx += THREADS) {
                    const int a0 = upper ? idx % kb : idx % nrow;
                    const int a1 = upper ? idx / kb : idx / nrow;
                    const int t = upper ? a1 : a0, c = upper ? a0 : a1;
                    S.set(rb + t, j0 + c, sW[t * LDP + c]);
                }
                __syncthreads();
            }
            // ---------------------------------------------- 3. trailing update (lower tiles)
            const int mt = n - m0;
            if (mt <= 0) continue;
            const int ntile = (mt + TB - 1) / TB;
            T *sI = sW;
            T *sK = sW + NB * LDT;
            // a thread owns a 4 x 4 block (row group ti, column group tk) of the 64 x 64 tile; warp
            // w owns rows 16*(w%4) .. +15 and columns 32*(w/4) .. +31, so a warp whose whole patch
            // lies above a diagonal tile's diagonal or past the matrix's last row or column skips
            // the tile (2 of 8 warps on every diagonal tile; the half-empty last row of tiles when
            // the trailing order is an odd multiple of 32). Inside the warp the index that is
            // contiguous in memory varies fastest across lanes (Lower: rows; Upper: columns of S)
            const int wrp = tid >> 5, ln = tid & 31;
            const int rg = wrp & 3, cg = wrp >> 2;
            const int ti = 4 * rg + (upper ? ln / 8 : ln % 4);    // row group (4 rows)
            const int tk = 8 * cg + (upper ? ln % 8 : ln / 4);    // column group (4 columns)
            for (int bi = 0; bi < ntile; ++bi) {
                const int I0 = m0 + bi * TB;
                for (int bk = 0; bk <= bi; ++bk) {
                    const int K0 = m0 + bk * TB;
                    const bool idle = I0 + 16 * rg >= n || K0 + 32 * cg >= n || (bi == bk && 16 * rg + 15 < 32 * cg);
                    for (int idx = tid; idx < kb * TB; idx += THREADS) {
                        const int a0 = upper ? idx % kb : idx % TB;
                        const int a1 = upper ? idx / kb : idx / TB;
                        const int rr = upper ? a1 : a0, c = upper ? a0 : a1;
                        sI[c * LDT + rr] = (I0 + rr < n) ? S.get(I0 + rr, j0 + c) : zero<T>();
                        sK[c * LDT + rr] = (K0 + rr < n) ? S.get(K0 + rr, j0 + c) : zero<T>();
                    }
                    __syncthreads();
                    if (!idle) {                  // warp-uniform: skip a wholly masked patch
                        T acc[4][4];
#pragma unroll
                        for (int a = 0; a < 4; ++a)
#pragma unroll
                            for (int b = 0; b < 4; ++b) acc[a][b] = zero<T>();
                        for (int c = 0; c < kb; ++c) {
                            T u[4], v[4];
#pragma unroll
                            for (int a = 0; a < 4; ++a) u[a] = sI[c * LDT + 4 * ti + a];
#pragma unroll
                            for (int b = 0; b < 4; ++b) v[b] = sK[c * LDT + 4 * tk + b];
#pragma unroll
                            for (int a = 0; a < 4; ++a)
#pragma unroll
                                for (int b = 0; b < 4; ++b) sub_mul_conj(acc[a][b], u[a], v[b]);
                        }
                        // acc = -L21_I L21_K^H; add into the trailing matrix, lower part only
#pragma unroll
                        for (int b = 0; b < 4; ++b)
#pragma unroll
                            for (int a = 0; a < 4; ++a) {
                                const int i = I0 + 4 * ti + a, k = K0 + 4 * tk + b;
                                if (i < n && k < n && i >= k) {
                                    T v = S.get(i, k);
                                    add_into(v, acc[a][b]);   // acc holds -sum
                                    S.set(i, k, v);
                                }
                            }
                    }
                    __syncthreads();
                }
            }
        }
        if (tid == 0 && !s_fail) args.info[mat] = 0;
        __syncthreads();
    }
    // ---------------------------------------------- solves (posv after success, potrs)
    if (mode != MODE_POTRF && !s_fail) {
        const int nrhs = args.nrhs;
        T *B = static_cast<T *>(args.B) + mat * args.stride_b;
        const int64_t ldb = args.ldb;
        // forward: L y = b
        for (int j = 0; j < n; ++j) {
            const R rl = R(1) / re(S.get(j, j));
            for (int c = tid; c < nrhs; c += THREADS) B[c * ldb + j] = scale(B[c * ldb + j], rl);
            __syncthreads();
            const int m = n - j - 1;
            for (int idx = tid; idx < m * nrhs; idx += THREADS) {
                const int r = j + 1 + idx % m, c = idx / m;
                sub_mul(B[c * ldb + r], S.get(r, j), B[c * ldb + j]);
            }
            __syncthreads();
        }
        // back: L^H x = y
        for (int i = n - 1; i >= 0; --i) {
            const R rl = R(1) / re(S.get(i, i));
            for (int c = tid; c < nrhs; c += THREADS) B[c * ldb + i] = scale(B[c * ldb + i], rl);
            __syncthreads();
            for (int idx = tid; idx < i * nrhs; idx += THREADS) {
                const int r = idx % i, c = idx / i;
                sub_mul(B[c * ldb + r], conj(S.get(i, r)), B[c * ldb + i]);
            }
            __syncthreads();
        }
    }
}

}  // namespace bl
