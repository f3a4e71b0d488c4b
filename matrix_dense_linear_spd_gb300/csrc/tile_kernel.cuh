// Register-tile Cholesky family ("tile"): the whole matrix lives in registers, spread over a
// P x P grid of threads in a 2-D cyclic layout, so every thread keeps a working share as the
// trailing matrix shrinks.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page; tiers "tiny" and "cta" are the prior art):
// right-looking Cholesky, one column j at a time:
//   pivot   d = A(j,j) (already updated by the earlier columns); fail if !(d > 0), first failure
//           wins and is reported 1-based ("potrf: correctness findings" item 6);
//   scale   L(j,j) = sqrt(d), L(i,j) = A(i,j) / sqrt(d) for i > j;
//   update  A(i,k) -= L(i,j) * conj(L(k,j)) for j < k <= i (lower triangle only).
// Upper runs the same recurrence on S(i,c) = conj(A(c,i)) ("can_run() terms": Upper is a load
// and store transform).
//
// Layout: thread (p, q) of a matrix owns rows i = p + P*s and columns k = q + P*t
// (s, t < S), i.e. tile entry a[s][t] = A(i, k); only s >= t is ever live. Thread index within
// the matrix is q*P + p, so the P owners of one column are adjacent lanes of one warp and the
// pivot reaches them with one shuffle. Each column is published once through shared memory
// (double-buffered, one barrier per column).
//
// posv ("The fused potrs solve"): the right-hand sides ride along as extra rows at the bottom
// of the tile, holding conj(B)^T. Factoring [A; B^H] column by column leaves those rows equal
// to (L^{-1} B)^H, i.e. the forward substitution L*Y = B comes out of the factorisation
// itself. A backward sweep over the rows of L then applies L^{-H}. Extra row c sits at tile row
// N-1-c, which is in block s = S-1 for every c < P, so all register indices stay static.
// potrs (solve only) runs the same sweeps with the factor loaded instead of computed.
#pragma once

#include "bl_types.cuh"

namespace bl {

template <typename T, int P, int S>
struct TileCfg {
    static constexpr int N = P * S;                     // capacity: n + nrhs <= N, nrhs <= P
    static constexpr int TPM = P * P;                   // threads per matrix
    static constexpr int G = TPM >= 128 ? 1 : 128 / TPM;  // matrices per CTA
    static constexpr int THREADS = G * TPM;
    static constexpr int CS = (S % 2) ? S : S + 1;      // column-buffer stride (odd: no conflicts)
    static constexpr int LDST = (N % 2) ? N : N + 1;    // staging leading dimension (odd)
    static constexpr bool WARP_SYNC = TPM <= 32;        // a matrix never spans two warps
    using R = real_t<T>;

    // dynamic shared memory layout (byte offsets), identical on host and device
    static constexpr size_t off_stage = 0;
    static constexpr size_t off_col = off_stage + sizeof(T) * G * P * LDST;
    static constexpr size_t off_x = off_col + sizeof(T) * 2 * G * P * CS;
    static constexpr size_t off_rs = off_x + sizeof(T) * 2 * G * P;
    static constexpr size_t off_info = off_rs + sizeof(R) * G * N;
    // second staging buffer: the load copies block b+1 while block b is distributed
    static constexpr size_t off_stage1 = ((off_info + sizeof(int) * G) + 15) / 16 * 16;
    static constexpr size_t smem_bytes = off_stage1 + sizeof(T) * G * P * LDST;
};

template <bool WARP>
__device__ __forceinline__ void tile_sync() {
    if (WARP) __syncwarp(); else __syncthreads();
}

// Issue the copies of staging block b (P columns of A, or P rows of S = columns of A for Upper)
// into buffer b & 1 as element-wise cp.async, and close one commit group (empty past the
// matrix). RT threads walk a column, CT columns at a time; thread (sr, sc) of the matrix.
template <typename T, int P, int RT, int CT, int LDST>
__device__ __forceinline__ void tile_issue(int b, bool live, bool upper, int n, int64_t lda, const T *A, T *stage0,
                                           T *stage1, int sr, int sc) {
    const int c0 = b * P;
    T *buf = (b & 1) ? stage1 : stage0;
    if (live && c0 < n) {
        if (!upper) {
            // columns c0..c0+P-1 of A, rows c..n-1 (lower part only)
            for (int cc = sc; cc < P; cc += CT) {
                const int c = c0 + cc;
                if (c >= n) break;
                for (int r = c + sr; r < n; r += RT)
                    cp_async_elem<sizeof(T)>(buf + cc * LDST + r, A + static_cast<int64_t>(c) * lda + r);
            }
        } else {
            // rows c0..c0+P-1 of S = columns of A, A rows 0..i (upper part only)
            for (int ii = sc; ii < P; ii += CT) {
                const int i = c0 + ii;
                if (i >= n) break;
                for (int k = sr; k <= i; k += RT)
                    cp_async_elem<sizeof(T)>(buf + ii * LDST + k, A + static_cast<int64_t>(i) * lda + k);
            }
        }
    }
    cp_async_commit();
}

template <typename T, int P, int S>
__global__ void __launch_bounds__(TileCfg<T, P, S>::THREADS)
tile_kernel(const BatchArgs args) {
    using C = TileCfg<T, P, S>;
    using R = typename C::R;
    constexpr int N = C::N, TPM = C::TPM, G = C::G, CS = C::CS, LDST = C::LDST;
    constexpr bool WS = C::WARP_SYNC;

    extern __shared__ __align__(16) unsigned char smem[];
    T *stage_all = reinterpret_cast<T *>(smem + C::off_stage);
    T *col_all = reinterpret_cast<T *>(smem + C::off_col);
    T *x_all = reinterpret_cast<T *>(smem + C::off_x);
    R *rs_all = reinterpret_cast<R *>(smem + C::off_rs);
    int *info_all = reinterpret_cast<int *>(smem + C::off_info);

    const int tid = threadIdx.x;
    const int g = tid / TPM;
    const int tl = tid - g * TPM;
    const int p = tl % P;
    const int q = tl / P;
    const int64_t mat = static_cast<int64_t>(blockIdx.x) * G + g;
    const bool live = mat < args.batch;
    const int n = args.n;
    const int mode = args.mode;
    const bool upper = args.upper != 0;
    const int nrhs = (mode == MODE_POTRF) ? 0 : args.nrhs;
    const int64_t lda = args.lda;
    T *A = static_cast<T *>(args.A) + (live ? mat * args.stride_a : 0);
    T *B = (mode == MODE_POTRF) ? nullptr
                                : static_cast<T *>(args.B) + (live ? mat * args.stride_b : 0);
    T *stage = stage_all + g * P * LDST;
    R *rsv = rs_all + g * N;
    // this thread's extra (right-hand-side) row, if any: tile row N-1-c lives at s = S-1, p = P-1-c
    const bool xrow = p >= P - nrhs;
    const int xc = P - 1 - p;
    // staging copy geometry: RT threads walk a column, CT columns at a time
    constexpr int RT = TPM < 32 ? TPM : 32;
    constexpr int CT = TPM / RT;
    const int sr = tl % RT, sc = tl / RT;

    T a[S][S];
#pragma unroll
    for (int s = 0; s < S; ++s)
#pragma unroll
        for (int t = 0; t <= s; ++t) a[s][t] = zero<T>();

    if (tl == 0) info_all[g] = 0;

    // ------------------------------------------------------------------ load A (staged)
    // Block b (P columns of A, or P rows of S for Upper) moves by element-wise cp.async into one
    // of two staging buffers, every copy of the block in flight at once and no register round
    // trip; block b+1 is issued before block b is distributed into the tile, so its HBM latency
    // overlaps that work. One commit group per block (empty past the matrix), waited for with
    // one group still in flight.
    T *const stage1 = reinterpret_cast<T *>(smem + C::off_stage1) + g * P * LDST;
    const bool do_load = live;
    tile_issue<T, P, RT, CT, LDST>(0, do_load, upper, n, lda, A, stage, stage1, sr, sc);
#pragma unroll
    for (int b = 0; b < S; ++b) {
        const int c0 = b * P;
        if (c0 >= n) break;
        tile_issue<T, P, RT, CT, LDST>(b + 1, do_load, upper, n, lda, A, stage, stage1, sr, sc);
        cp_async_wait_group<1>();
        tile_sync<WS>();
        const T *buf = (b & 1) ? stage1 : stage;
        if (!upper) {
            const int c = c0 + q;
#pragma unroll
            for (int s = b; s < S; ++s) {
                const int i = p + P * s;
                if (c < n && i < n && (s > b || p >= q)) a[s][b] = buf[q * LDST + i];
            }
        } else {
            const int i = c0 + p;
#pragma unroll
            for (int t = 0; t <= b; ++t) {
                const int k = q + P * t;
                if (i < n && (t < b || q <= p)) a[b][t] = conj(buf[p * LDST + k]);
            }
        }
        tile_sync<WS>();
    }
    cp_async_wait_all();
    // right-hand sides as conjugated extra rows: entry (N-1-c, k) = conj(B(k, c))
    if (nrhs > 0 && live && xrow) {
#pragma unroll
        for (int t = 0; t < S; ++t) {
            const int k = q + P * t;
            if (k < n) a[S - 1][t] = conj(B[static_cast<int64_t>(xc) * args.ldb + k]);
        }
    }

    // ------------------------------------------------------------------ factor / forward sweep
#pragma unroll
    for (int T0 = 0; T0 < S; ++T0) {
        if (T0 * P >= n) break;
        for (int jj = 0; jj < P; ++jj) {
            const int j = T0 * P + jj;
            if (j >= n) break;
            T *col = col_all + ((j & 1) * G + g) * P * CS;
            const int src = (g * TPM + jj * P + jj) & 31;
            const R d = __shfl_sync(0xffffffffu, re(a[T0][T0]), src);
            const bool owner = (q == jj);
            if (mode != MODE_POTRS) {
                const bool ok = d > R(0);
                const R rs = ok ? rsqrt_of(d) : R(0);
                const R ljj = ok ? d * rs : d;
                if (owner) {
#pragma unroll
                    for (int s = T0; s < S; ++s) {
                        if (s > T0 || p >= jj) {
                            T v = a[s][T0];
                            v = (s == T0 && p == jj) ? from_real<T>(ljj) : scale(v, rs);
                            a[s][T0] = v;
                            col[p * CS + s] = v;
                        }
                    }
                    if (p == jj) {
                        rsv[j] = rs;
                        if (!ok && info_all[g] == 0) info_all[g] = j + 1;
                    }
                }
            } else {
                const R rs = R(1) / d;
                if (owner) {
#pragma unroll
                    for (int s = T0; s < S; ++s) {
                        if (s > T0 || p >= jj) {
                            T v = a[s][T0];
                            if (s == S - 1 && xrow) v = scale(v, rs);
                            a[s][T0] = v;
                            col[p * CS + s] = v;
                        }
                    }
                    if (p == jj) rsv[j] = rs;
                }
            }
            tile_sync<WS>();
            T lr[S], lc[S];
#pragma unroll
            for (int s = T0; s < S; ++s) {
                lr[s] = col[p * CS + s];
                lc[s] = col[q * CS + s];
            }
            if (mode != MODE_POTRS) {
#pragma unroll
                for (int s = T0; s < S; ++s)
#pragma unroll
                    for (int t = T0; t <= s; ++t) {
                        const bool pred = (t > T0 || q > jj) && (s > t || p >= q);
                        if (pred) sub_mul_conj(a[s][t], lr[s], lc[t]);
                    }
            } else if (xrow) {
#pragma unroll
                for (int t = T0; t < S; ++t) {
                    const bool pred = (t > T0 || q > jj) && (S - 1 > t || p >= q);
                    if (pred) sub_mul_conj(a[S - 1][t], lr[S - 1], lc[t]);
                }
            }
        }
    }

    // ------------------------------------------------------------------ backward sweep (L^H)
    if (nrhs > 0) {
#pragma unroll
        for (int T0 = S - 1; T0 >= 0; --T0) {
            if (T0 * P >= n) continue;
            for (int jj = P - 1; jj >= 0; --jj) {
                const int i = T0 * P + jj;
                if (i >= n) continue;
                // parity offset by one so the first backward step never reuses the buffer the
                // last forward step is still reading
                const int buf = (i + 1) & 1;
                T *row = col_all + (buf * G + g) * P * CS;
                T *xb = x_all + (buf * G + g) * P;
                if (xrow && q == jj) {
                    const T x = scale(a[S - 1][T0], rsv[i]);
                    a[S - 1][T0] = x;
                    xb[xc] = x;
                }
                if (p == jj) {
#pragma unroll
                    for (int t = 0; t <= T0; ++t)
                        if (t < T0 || q < jj) row[q * CS + t] = a[T0][t];
                }
                tile_sync<WS>();
                if (xrow) {
                    const T x = xb[xc];
#pragma unroll
                    for (int t = 0; t <= T0; ++t)
                        if (t < T0 || q < jj) sub_mul(a[S - 1][t], row[q * CS + t], x);
                }
            }
        }
    }

    tile_sync<WS>();
    // ------------------------------------------------------------------ store the factor
    if (mode != MODE_POTRS) {
#pragma unroll
        for (int b = 0; b < S; ++b) {
            const int c0 = b * P;
            if (c0 >= n) break;
            if (!upper) {
                const int c = c0 + q;
#pragma unroll
                for (int s = b; s < S; ++s) {
                    const int i = p + P * s;
                    if (c < n && i < n && (s > b || p >= q)) stage[q * LDST + i] = a[s][b];
                }
                tile_sync<WS>();
                if (live)
                    for (int cc = sc; cc < P; cc += CT) {
                        const int cg = c0 + cc;
                        if (cg >= n) break;
                        for (int r = cg + sr; r < n; r += RT) A[static_cast<int64_t>(cg) * lda + r] = stage[cc * LDST + r];
                    }
            } else {
                const int i = c0 + p;
#pragma unroll
                for (int t = 0; t <= b; ++t) {
                    const int k = q + P * t;
                    if (i < n && (t < b || q <= p)) stage[p * LDST + k] = conj(a[b][t]);
                }
                tile_sync<WS>();
                if (live)
                    for (int ii = sc; ii < P; ii += CT) {
                        const int ig = c0 + ii;
                        if (ig >= n) break;
                        for (int k = sr; k <= ig; k += RT) A[static_cast<int64_t>(ig) * lda + k] = stage[ii * LDST + k];
                    }
            }
            tile_sync<WS>();
        }
        if (live && tl == 0) args.info[mat] = info_all[g];
    }
    // ------------------------------------------------------------------ store X (success only)
    // A solve-only pass that follows a posv pass is given info and skips the failed items.
    const bool solved = (mode == MODE_POTRS) ? (args.info == nullptr || !live || args.info[mat] == 0)
                                             : (info_all[g] == 0);
    if (nrhs > 0 && live && xrow && solved) {
#pragma unroll
        for (int t = 0; t < S; ++t) {
            const int k = q + P * t;
            if (k < n) B[static_cast<int64_t>(xc) * args.ldb + k] = conj(a[S - 1][t]);
        }
    }
}

}  // namespace bl
