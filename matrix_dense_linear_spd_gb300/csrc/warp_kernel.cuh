// Lane-row Cholesky family ("warp"): one matrix per P lanes of a warp (G = 32/P matrices per
// warp), each lane holding R rows in registers, for n <= P*R <= 32.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "potrf: the tiny tier": lanes own
// rows in registers, cross-lane values go by shuffles, no barriers beyond the warp): right-looking
// Cholesky one column j at a time -- pivot d = A(j,j) from its owner lane by one shuffle, fail if
// !(d > 0) (first failure wins, info = j+1), L(j,j) = sqrt(d), L(i,j) = A(i,j)*rsqrt(d),
// then A(i,k) -= L(i,j)*conj(L(k,j)) for j < k <= i.
//
// GB300 layout:
//  * lane l of a partition owns rows i = l + P*rho (rho < R), cyclic, so every lane keeps
//    trailing work as the matrix shrinks; with R > 1 one warp instruction advances G matrices;
//  * the column L(:,j) is published once per step into a double-buffered per-partition slot in
//    shared memory and read back as 16-byte broadcast loads (one load serves E entries for all
//    lanes), far fewer instructions than one shuffle per entry;
//  * warps are persistent: while a warp factors its current group of G matrices, the next
//    group's referenced triangle is already streaming into a compacted shared-memory slab by
//    cp.async (16-byte chunks when the layout is 16-byte aligned, element copies otherwise), so
//    HBM latency overlaps compute and no registers are tied up by loads in flight. The slab
//    holds, per matrix, only the chunks that intersect the referenced triangle, and its
//    per-matrix stride is padded so the partitions of a warp read disjoint banks.
//
// posv / potrs (same page, "The fused posv tier" and "posv: the backward solve costs a
// transpose"): up to RHS right-hand sides per pass live in registers next to the rows. The
// forward solve L*y = b runs inside the column loop (once column j is scaled, y_j = b_j/L(j,j)
// is broadcast and rows below subtract L(i,j)*y_j). The backward solve L^H*x = y needs row i of
// L, which only its owner lane holds: each block of P rows is written once into a staging slab
// (the transpose through shared memory) and the sweep reads conj(L(i,r)) from there. The
// solve-capable instantiation is separate, so the factor-only kernel keeps its registers.
#pragma once

#include "bl_types.cuh"

namespace bl {

// Compacted per-matrix slab for an N x N item, in chunks of E elements (16 bytes).
//   Lower: column c keeps rows [E*floor(c/E), N)        (the chunks meeting rows >= c)
//   Upper: column c keeps rows [0, E*ceil((c+1)/E))     (the chunks meeting rows <= c)
template <int N, int E>
struct TriSlab {
    __host__ __device__ static constexpr int lo_first(int c) { return (c / E) * E; }
    __host__ __device__ static constexpr int lo_len(int c) { return N - lo_first(c); }
    __host__ __device__ static constexpr int lo_off(int c) {
        int o = 0;
        for (int x = 0; x < c; ++x) o += lo_len(x);
        return o;
    }
    __host__ __device__ static constexpr int up_len(int c) { return ((c + E) / E) * E; }
    __host__ __device__ static constexpr int up_off(int c) {
        int o = 0;
        for (int x = 0; x < c; ++x) o += up_len(x);
        return o;
    }
    static constexpr int size = lo_off(N) > up_off(N) ? lo_off(N) : up_off(N);
};

// Upper slab offset of column i at run time: sum_{x < i} E*ceil((x+1)/E)
//   = E*(i + E*m*(m-1)/2 + m*r) with m = floor(i/E), r = i - m*E.
__device__ __forceinline__ int upper_slab_offset(int i, int E) {
    const int m = i / E, r = i - m * E;
    return E * (i + E * m * (m - 1) / 2 + m * r);
}

template <typename T, int P, int R>
struct WarpCfg {
    static constexpr int N = P * R;
    // registers (32-bit words) one lane spends on its rows
    static constexpr int row_words() {
        int w = 0;
        for (int r = 0; r < R; ++r) w += (P * r + P) * static_cast<int>(sizeof(T) / 4);
        return w;
    }
    // right-hand sides per solve pass: as many as fit next to the rows without spilling
    static constexpr int RHS = row_words() <= 48 ? 8 : (row_words() <= 96 ? 4 : 2);
    static constexpr int G = 32 / P;                 // matrices per warp
    static constexpr int WARPS = 4;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int PER_CTA = G * WARPS;
    static constexpr int E = 16 / static_cast<int>(sizeof(T));   // elements per 16 bytes
    static_assert(N % E == 0, "N must be a multiple of the 16-byte chunk");
    static constexpr int CB = N;                     // column-buffer length
    static constexpr int RB = (RHS + E - 1) / E * E; // broadcast slots for y_j (16-byte multiple)
    static constexpr int CBX = CB + RB;
    // per-partition column slots (two buffers): stride congruent to P modulo the bank cycle, so
    // the partitions of a warp store their columns into disjoint banks
    static constexpr int col_stride() {
        int s = 2 * CBX;
        while (((s - P) % (128 / static_cast<int>(sizeof(T))) + 128 / static_cast<int>(sizeof(T))) %
                   (128 / static_cast<int>(sizeof(T))) != 0)
            s += E;
        return s;
    }
    static constexpr int COLS = col_stride();
    static constexpr int LDU = ((N + 1) % 2) ? N + 1 : N + 2;  // staging leading dim (odd)
    // per-matrix slab stride: >= the slab, a multiple of E, and congruent to P modulo one bank
    // cycle (128 bytes), so partition g of a warp starts g*P elements into the bank cycle
    static constexpr int BANKCYC = 128 / static_cast<int>(sizeof(T));
    static constexpr int slab_stride() {
        int s = (TriSlab<N, E>::size + E - 1) / E * E;
        while (((s - P) % BANKCYC + BANKCYC) % BANKCYC != 0) s += E;
        return s;
    }
    static constexpr int MSTRIDE = slab_stride();
    static constexpr int SLOTS = G * WARPS;
    static constexpr size_t tri_bytes = sizeof(T) * MSTRIDE * SLOTS;
    static constexpr size_t col_bytes = sizeof(T) * COLS * SLOTS;
    static constexpr size_t stage_bytes = sizeof(T) * P * LDU * SLOTS;
    static constexpr size_t off_col = (tri_bytes + 15) / 16 * 16;
    static constexpr size_t off_stage = off_col + (col_bytes + 15) / 16 * 16;
    static constexpr size_t off_rs = off_stage + (stage_bytes + 15) / 16 * 16;
    static constexpr size_t rs_bytes = sizeof(real_t<T>) * N * SLOTS;
    static constexpr size_t off_x = off_rs + (rs_bytes + 15) / 16 * 16;
    static constexpr size_t x_bytes = sizeof(T) * 2 * RB * SLOTS;
    static constexpr size_t smem_lower = off_stage;               // Lower potrf: no staging slab
    // full-square slabs (items stored back to back, n = N): each matrix copied whole. Lower keeps
    // the column stride N (the copy is one contiguous run per matrix); Upper pads each column by
    // 16 bytes so a row of S (a column of A) reads in 16-byte pieces across 8 lanes without bank
    // conflicts. The matrix stride is congruent to P modulo one bank cycle (the warp's
    // partitions read disjoint banks).
    static constexpr int NS_L = N;
    static constexpr int NS = N + E;
    static constexpr int FSTRIDE = N * NS + ((P - (N * NS) % BANKCYC) % BANKCYC + BANKCYC) % BANKCYC;
    static constexpr size_t full_bytes = sizeof(T) * FSTRIDE * SLOTS;
    static constexpr size_t off_col_full = (full_bytes + 15) / 16 * 16;
    static constexpr size_t smem_full = off_col_full + (col_bytes + 15) / 16 * 16;
    static constexpr bool full_ok = sizeof(T) <= 8 && (N * N / E) % 32 == 0 && (P * sizeof(T)) % 16 == 0 &&
                                    (FSTRIDE * sizeof(T)) % 16 == 0;
    // the solve kernel on whole squares keeps the rows, the right-hand sides and the slab
    // addresses live at once; above 128 words of rows per lane it no longer fits 255 registers
    // (ptxas spills), so those geometries solve from the compacted slab
    static constexpr bool full_solve_ok = full_ok && row_words() <= 128;
    static constexpr size_t smem_potrf = off_stage + stage_bytes;
    static constexpr size_t smem_solve = off_x + x_bytes;
    static constexpr size_t full_shift = off_col_full - off_col;   // solve areas move up by this
    static constexpr size_t smem_solve_full = smem_solve + full_shift;
    static constexpr size_t smem_potrf_full = smem_potrf + full_shift;   // Upper: with the staging slab
    // launch bound for the factor-only kernel: registers held by the rows (32-bit words) plus
    // about 45 for addresses and temporaries, rounded down to whole CTAs per SM
    static constexpr int min_blocks() {
        const int m = 65536 / (THREADS * (row_words() + 45));
        return m < 1 ? 1 : (m > 8 ? 8 : m);
    }
    // complex factor-only kernels on whole squares keep the 16-byte row reads of the pick live
    // longer: one CTA per SM fewer than min_blocks() (ptxas spills otherwise)
    static constexpr int min_blocks_full() {
        const int m = min_blocks() - (is_cplx<T>::value ? 1 : 0);
        return m < 1 ? 1 : m;
    }
    // solve kernels: the rows, the right-hand-side registers (R x RHS words per lane) and about 70
    // for addresses, the broadcast solution values and temporaries (ptxas: no spill at this
    // bound for the f32 geometries; the shared-memory footprint may still cap residency lower)
    static constexpr int min_blocks_solve(size_t smem) {
        const int m = 65536 / (THREADS * (row_words() + R * RHS * static_cast<int>(sizeof(T) / 4) + 70));
        const int by_smem = static_cast<int>(233472 / (smem + 1024));    // 228 KB per SM, 1 KB per CTA reserved
        const int b = m < by_smem ? m : by_smem;
        return b < 1 ? 1 : (b > 8 ? 8 : b);
    }
    // the packed update keeps column pairs in aligned register pairs: about 15 more per lane
    static constexpr int min_blocks_packed() {
        const int m = 65536 / (THREADS * (row_words() + 60));
        return m < 1 ? 1 : (m > 8 ? 8 : m);
    }
    // float2-row kernels on compacted slabs: the rows are their own register pairs, about 48 more
    // for addresses, the column pieces in flight and the pivot chain
    static constexpr int min_blocks_v2c() {
        const int m = 65536 / (THREADS * (row_words() + 48));
        return m < 1 ? 1 : (m > 8 ? 8 : m);
    }
    static constexpr int blocks_by_smem(size_t bytes) { return static_cast<int>(233472 / (bytes + 1024)); }
    // the float2-row kernel takes the compacted slab when whole-square slabs would hold fewer CTAs
    // per SM than its registers allow and one sweep of 32 lanes spans E whole columns
    static constexpr bool v2_compact = sizeof(T) == 4 && N / E > 0 && 32 % (N / E) == 0 && 32 / (N / E) == E &&
                                       (N * N / E) % 32 == 0 && blocks_by_smem(smem_full) < min_blocks_v2c();
};

template <typename T>
struct alignas(16) Vec16 {
    T v[16 / sizeof(T)];
};

// Closed forms of the slab offsets for run-time column indices.
template <int N, int E>
__device__ __forceinline__ int lower_slab_offset(int c) {
    // sum_{x < c} (N - E*floor(x/E)) = c*N - E*(E*m*(m-1)/2 + m*r), m = floor(c/E), r = c - m*E
    const int m = c / E, r = c - m * E;
    return c * N - E * (E * m * (m - 1) / 2 + m * r);
}

// Copy one group's contiguous run of whole squares into the slab with column stride NS: chunk k
// (16 bytes) is matrix k / CPM, column (k mod CPM) / CPCOL, chunk k mod CPCOL of that column.
// Only the chunks that meet the referenced triangle move (Lower: chunk q of column c when it
// holds a row >= c; Upper: when it holds a row <= c), so HBM delivers the triangle's sectors and
// not the whole square; the slab positions of the other chunks keep stale values, which only
// reach register entries on the other side of the diagonal (never read into the factor).
// When 32 lanes span whole columns every offset but the lane's is an immediate.
template <typename T, bool UPPER, int NS, int CPM, int CPCOL, int IT, int FSTRIDE, int E>
__device__ __forceinline__ void full_copy(T *tri, const T *src, int lane, int64_t mleft) {
    if constexpr (32 % CPCOL == 0) {
        T *dst = tri + (lane / CPCOL) * NS + (lane % CPCOL) * E;
        // the lane's chunk q = lane % CPCOL in column c = c0 + lane / CPCOL is needed when
        // (Lower) q*E + E - 1 >= c, i.e. c0 <= dl, or (Upper) q*E <= c, i.e. c0 >= du
        const int dl = (lane % CPCOL) * E + E - 1 - lane / CPCOL;
        const int du = (lane % CPCOL) * E - lane / CPCOL;
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int gg = (32 * it) / CPM;
            const int c0 = (32 * it - gg * CPM) / CPCOL;
            const bool need = UPPER ? (c0 >= du) : (c0 <= dl);
            if (gg < mleft && need) cp_async_16(dst + gg * FSTRIDE + c0 * NS, src + 32 * it * E);
        }
    } else {
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int k = lane + 32 * it;
            const int gg = k / CPM, w = k - gg * CPM, c = w / CPCOL, q = w - c * CPCOL;
            const bool need = UPPER ? (q * E <= c) : (q * E + E - 1 >= c);
            if (gg < mleft && need) cp_async_16(tri + gg * FSTRIDE + c * NS + q * E, src + 32 * it * E);
        }
    }
}

// Issue the asynchronous copy of group `grp`'s referenced triangles into the warp's slab.
// Lanes map to fixed (matrix, chunk) or (matrix, row) pairs and sweep the columns, so the copy
// costs a handful of registers, not one address per chunk; 16-byte chunks when the layout
// allows them, element copies otherwise.
template <typename T, int P, int R, bool FULL = false>
__device__ __forceinline__ void warp_prefetch(const BatchArgs &args, T *tri, int64_t grp, int lane, bool vec) {
    using C = WarpCfg<T, P, R>;
    constexpr int N = C::N, G = C::G, E = C::E, MS = C::MSTRIDE;
    const int n = args.n;
    const int64_t lda = args.lda, sa = args.stride_a;
    const bool upper = args.upper != 0;
    const T *A0 = static_cast<const T *>(args.A) + grp * G * sa;
    const int64_t mleft = args.batch - grp * G;            // live matrices in this group
    if constexpr (FULL) {
        // the group's items are one contiguous run of G*N*N elements
        constexpr int CPM = N * N / E;                     // chunks per matrix
        constexpr int CPCOL = N / E;                       // chunks per column
        constexpr int IT = G * CPM / 32;
        static_assert((G * CPM) % 32 == 0 && CPM % 32 == 0, "whole chunks per lane");
        const T *src = A0 + lane * E;
        if (upper) full_copy<T, true, C::NS, CPM, CPCOL, IT, C::FSTRIDE, E>(tri, src, lane, mleft);
        else full_copy<T, false, C::NS_L, CPM, CPCOL, IT, C::FSTRIDE, E>(tri, src, lane, mleft);
        cp_async_commit();
        return;
    }
    if (vec) {
        // lanes map to fixed (matrix, 16-byte chunk) pairs; the column loop is unrolled so every
        // slab offset is a compile-time constant, the source is one running pointer per sweep,
        // and a lane's chunk takes part in the columns below one threshold (Lower: c < Q*E + E,
        // the chunk meets rows >= c) or from one threshold on (Upper: c >= Q*E)
        constexpr int NQ = N / E;                          // chunks per full column
        constexpr int CPC = G * NQ;                        // (matrix, chunk) pairs per column
        constexpr int ITC = (CPC + 31) / 32;               // lane sweeps per column
        const T *src[ITC];
        int dst[ITC], lim[ITC];
#pragma unroll
        for (int it = 0; it < ITC; ++it) {
            const int t = lane + 32 * it;
            const int gg = t / NQ, Q = t - gg * NQ;
            const bool ok = t < CPC && gg < mleft && Q * E < n;
            lim[it] = upper ? (ok ? Q * E : N) : (ok ? Q * E + E : 0);
            src[it] = A0 + gg * sa + Q * E;
            dst[it] = gg * MS + Q * E;
        }
        using L = TriSlab<N, E>;
        if (!upper) {
#pragma unroll
            for (int c = 0; c < N; ++c) {
                if (c >= n) break;
#pragma unroll
                for (int it = 0; it < ITC; ++it) {
                    if (c < lim[it]) cp_async_16(tri + dst[it] + (L::lo_off(c) - L::lo_first(c)), src[it]);
                    src[it] += lda;
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < N; ++c) {
                if (c >= n) break;
#pragma unroll
                for (int it = 0; it < ITC; ++it) {
                    if (c >= lim[it]) cp_async_16(tri + dst[it] + L::up_off(c), src[it]);
                    src[it] += lda;
                }
            }
        }
    } else {
        // element copies (any alignment): Lower rows c..n-1, Upper rows 0..c of column c
        constexpr int EPC = G * N;                         // (matrix, row) pairs per column
        constexpr int ITER = (EPC + 31) / 32;
        for (int c = 0; c < n; ++c) {
#pragma unroll
            for (int it = 0; it < ITER; ++it) {
                const int t = lane + 32 * it;
                const int gg = t / N, r = t - gg * N;
                if (t >= EPC || gg >= mleft || r >= n) continue;
                int pos;
                if (!upper) {
                    if (r < c) continue;
                    pos = lower_slab_offset<N, E>(c) + r - (c / E) * E;
                } else {
                    if (r > c) continue;
                    pos = upper_slab_offset(c, E) + r;
                }
                cp_async_elem<sizeof(T)>(tri + gg * MS + pos, A0 + gg * sa + c * lda + r);
            }
        }
    }
    cp_async_commit();
}

// PK (f32 only): the rank-1 update runs on column pairs (k, k+1) as packed two-lane FP32 FMAs
// (fma.rn.f32x2), one instruction per pair of entries of a row.
template <typename T, int P, int R, bool SOLVE, int MINB, bool FULL = false, bool PK = false>
__global__ void __launch_bounds__(128, MINB) warp_kernel(const BatchArgs args) {
    static_assert(!PK || (sizeof(T) == 4 && !is_cplx<T>::value && P % 2 == 0), "packed update: f32, even P");
    using C = WarpCfg<T, P, R>;
    using L = TriSlab<C::N, C::E>;
    using Rt = real_t<T>;
    constexpr int N = C::N, G = C::G, E = C::E, CB = C::CB, CBX = C::CBX, LDU = C::LDU, RHS = C::RHS;
    constexpr int RB = C::RB, MS = C::MSTRIDE;
    extern __shared__ __align__(16) unsigned char smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane / P;
    const int l_in = lane - g * P;
    const int slot = warp * G + g;
    const int n = args.n;
    const bool upper = args.upper != 0;
    const int64_t lda_in = args.lda;
    // the warp's slab (G matrices): compacted triangles, or whole squares (FULL)
    T *tri = reinterpret_cast<T *>(smem) + warp * G * (FULL ? C::FSTRIDE : MS);
    T *colbuf = reinterpret_cast<T *>(smem + (FULL ? C::off_col_full : C::off_col)) + slot * C::COLS;
    constexpr size_t shift = FULL ? C::full_shift : 0;
    T *stage = reinterpret_cast<T *>(smem + C::off_stage + shift) + slot * P * LDU;
    const int mode = SOLVE ? args.mode : MODE_POTRF;
    const bool factor = mode != MODE_POTRS;
    const int nrhs = SOLVE ? min(args.nrhs, RHS) : 0;
    Rt *rsb = SOLVE ? reinterpret_cast<Rt *>(smem + C::off_rs + shift) + slot * N : nullptr;
    T *xsb = SOLVE ? reinterpret_cast<T *>(smem + C::off_x + shift) + slot * 2 * RB : nullptr;

    // Identity padding: the slab positions of rows/columns >= n are never written by a prefetch,
    // so filling the whole slab with the identity once makes every later pick see an n x n item
    // bordered by the identity. The column loop then runs all N steps with no run-time bounds:
    // padding pivots are exactly 1 and padding entries stay 0.
    // (whole squares of n = N items need no padding)
    if (!FULL) {
        for (int t = lane; t < G * MS; t += 32) tri[t] = zero<T>();
        __syncwarp();
        for (int t = lane; t < G * N; t += 32) {
            const int gg = t / N, c = t - gg * N;
            const int pos = upper ? upper_slab_offset(c, E) + c : lower_slab_offset<N, E>(c) + c - (c / E) * E;
            tri[gg * MS + pos] = from_real<T>(Rt(1));
        }
        __syncwarp();
    }

    // 16-byte chunk copies need every column start 16-byte aligned and whole chunks inside n
    const bool vec = (n % E == 0) && ((lda_in * static_cast<int64_t>(sizeof(T))) % 16 == 0) &&
                     ((args.stride_a * static_cast<int64_t>(sizeof(T))) % 16 == 0) &&
                     ((reinterpret_cast<uintptr_t>(args.A) & 15) == 0);
    const int64_t ngroups = (args.batch + G - 1) / G;
    const int64_t gstep = static_cast<int64_t>(gridDim.x) * C::WARPS;
    int64_t grp = static_cast<int64_t>(blockIdx.x) * C::WARPS + warp;
    if (grp < ngroups) warp_prefetch<T, P, R, FULL>(args, tri, grp, lane, vec);

    for (; grp < ngroups; grp += gstep) {
        // Opaque copies of the lane index and leading dimension: without them the compiler
        // hoists every per-element address of the loop body out of this loop and keeps them
        // all live, which doubles the register count and halves occupancy.
        int l = l_in;
        int64_t lda = lda_in;
        asm volatile("" : "+r"(l));
        asm volatile("" : "+l"(lda));
        const int64_t mat = grp * G + g;
        const bool live = mat < args.batch;

        // -------------------------------------------------------------- pick from the slab
        T a[R][N];
        cp_async_wait_all();
        __syncwarp();
        const T *my = tri + g * (FULL ? C::FSTRIDE : MS);
        if (FULL && !upper) {
#pragma unroll
            for (int c = 0; c < N; ++c)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (P * r + P - 1 < c) continue;          // block r has no row >= c
                    a[r][c] = my[c * C::NS_L + l + P * r];
                }
        } else if (FULL) {
            // row i of S is column i of A: 16 bytes at a time, conjugated
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const T *rowp = my + (l + P * r) * C::NS;
#pragma unroll
                for (int c = 0; c < P * r + P; c += E) {
                    const Vec16<T> v = *reinterpret_cast<const Vec16<T> *>(rowp + c);
#pragma unroll
                    for (int e = 0; e < E; ++e) a[r][c + e] = conj(v.v[e]);
                }
            }
        } else if (!upper) {
#pragma unroll
            for (int c = 0; c < N; ++c)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (P * r + P - 1 < c) continue;          // block r has no row >= c
                    // rows i < c of the block read other entries of the slab: they land in the
                    // unused upper part of the lane's register row and never reach the factor
                    a[r][c] = my[L::lo_off(c) + l + P * r - L::lo_first(c)];
                }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int i = l + P * r;
                const T *rowp = my + upper_slab_offset(i, E);   // column i of A = row i of S
#pragma unroll
                for (int c = 0; c < P * r + P; ++c) a[r][c] = conj(rowp[c]);
            }
        }
        __syncwarp();
        if (grp + gstep < ngroups) warp_prefetch<T, P, R, FULL>(args, tri, grp + gstep, lane, vec);

        T *A = static_cast<T *>(args.A) + (live ? mat * args.stride_a : 0);
        T *B = SOLVE ? static_cast<T *>(args.B) + (live ? mat * args.stride_b : 0) : nullptr;
        // right-hand sides: b[r][c] = B(l + P*r, c), zero in the padding rows
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

        // -------------------------------------------------------------- factor (+ forward solve)
        unsigned failed = 0;                                   // bit j: pivot j was not positive
#pragma unroll
        for (int j = 0; j < N; ++j) {
            // columns >= n are identity padding: skipping them is exact, and the uniform branch
            // keeps the scheduler from interleaving all N unrolled steps (which costs registers)
            // n = N with whole squares: an empty asm fence replaces the exit test where the
            // registers allow (the scheduler may then overlap neighbouring columns a little)
            if (FULL && PK && (SOLVE || R <= 2)) {
                asm volatile("" ::: "memory");
            } else if (j >= n) {
                break;
            }
            const int rj = j / P, lj = j - rj * P;
            const Rt d = __shfl_sync(0xffffffffu, re(a[rj][j]), g * P + lj);
            T *col = colbuf + (j & 1) * CBX;
            Rt rs;
            if (factor) {
                const bool ok = d > Rt(0);
                rs = ok ? rsqrt_of(d) : Rt(0);
                failed |= ok ? 0u : (1u << j);
                // scale rows >= j (rows < j of block rj are unused upper entries: scaling them
                // is harmless). For a real type the diagonal comes out as d * (1/sqrt(d)) by the
                // same scaling; a complex diagonal is set to that real value (its imaginary part
                // is ignored). A failed pivot zeroes its column (the rest is unspecified).
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r < rj) continue;
                    T v = scale(a[r][j], rs);
                    if (is_cplx<T>::value && r == rj && l == lj) v = from_real<T>(d * rs);
                    a[r][j] = v;
                    col[l + P * r] = v;
                }
            } else {
                rs = Rt(1) / d;                                // the factor is given: 1 / L(j,j)
            }
            if (SOLVE) {
                // forward substitution, axpy form: y_j = b_j / L(j,j), then b_i -= L(i,j) y_j
                if (l == lj) {
#pragma unroll
                    for (int c = 0; c < RHS; ++c) {
                        b[rj][c] = scale(b[rj][c], rs);
                        col[CB + c] = b[rj][c];
                    }
                    rsb[j] = rs;
                }
            }
            __syncwarp();
            if (SOLVE) {
#pragma unroll
                for (int q = 0; q < RB / E; ++q) {
                    const Vec16<T> yv = reinterpret_cast<const Vec16<T> *>(col + CB)[q];
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int c = q * E + e;
                        if (c >= RHS) continue;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (P * r + P - 1 <= j) continue;      // no row > j in block r
                            const int i = l + P * r;
                            if (i > j) sub_mul(b[r][c], a[r][j], yv.v[e]);
                        }
                    }
                }
            }
            if (!factor) continue;
            if constexpr (PK) {
                // pairs (k, k+1), k even: both trailing -> one packed FMA; only k+1 trailing (k = j)
                // -> one scalar FMA. P is even, so a block with a row >= k also has one >= k+1.
                float2 m2[R];
#pragma unroll
                for (int r = 0; r < R; ++r) m2[r] = make_float2(-re(a[r][j]), -re(a[r][j]));
#pragma unroll
                for (int q = (j + 1) / E; q < CB / E; ++q) {
                    const Vec16<T> ck = reinterpret_cast<const Vec16<T> *>(col)[q];
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        const int k = q * E + e;
                        if (k + 1 <= j) continue;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (P * r + P - 1 < k) continue;   // no row >= k in block r
                            if (k <= j) {
                                sub_mul_conj(a[r][k + 1], a[r][j], ck.v[e + 1]);
                            } else {
                                const float2 t = __ffma2_rn(m2[r], make_float2(re(ck.v[e]), re(ck.v[e + 1])),
                                                            make_float2(re(a[r][k]), re(a[r][k + 1])));
                                a[r][k] = t.x;
                                a[r][k + 1] = t.y;
                            }
                        }
                    }
                }
            } else {
                // rank-1 update of the trailing rows/columns k > j, 16 bytes of the column at a time
#pragma unroll
                for (int q = (j + 1) / E; q < CB / E; ++q) {
                    const Vec16<T> ck = reinterpret_cast<const Vec16<T> *>(col)[q];
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int k = q * E + e;
                        if (k <= j) continue;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (P * r + P - 1 < k) continue;   // no row >= k in block r
                            sub_mul_conj(a[r][k], a[r][j], ck.v[e]);
                        }
                    }
                }
            }
        }
        const int info = failed ? (__ffs(failed)) : 0;         // first failing column, 1-based

        // -------------------------------------------------------------- backward solve
        if (SOLVE) {
            // L^H x = y, one block of P rows at a time from the bottom: the block's rows of L are
            // transposed through the staging slab, then x_i is broadcast and rows r < i subtract
            // conj(L(i,r)) x_i. Padding rows carry y = 0, so they contribute nothing.
#pragma unroll
            for (int rb = R - 1; rb >= 0; --rb) {
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
                    T *xs = xsb + (i & 1) * RB;
                    if (l == ii) {
                        const Rt ri = rsb[i];
#pragma unroll
                        for (int c = 0; c < RHS; ++c) {
                            b[rb][c] = scale(b[rb][c], ri);
                            xs[c] = b[rb][c];
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r <= rb; ++r) {
                        const int rr = l + P * r;
                        if (rr < i) {
                            const T lir = conj(stage[ii * LDU + rr]);
#pragma unroll
                            for (int c = 0; c < RHS; ++c) sub_mul(b[r][c], lir, xs[c]);
                        }
                    }
                }
            }
            __syncwarp();
        }

        // -------------------------------------------------------------- store
        // fresh opaque copies again, so the store's per-element predicates are not carried
        // (as live registers) all the way from the pick above
        asm volatile("" : "+r"(l));
        asm volatile("" : "+l"(lda));
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
            continue;
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
            // one running column pointer; a row block entirely at or below the diagonal needs
            // only its rows' bounds check
            bool row_ok[R];
#pragma unroll
            for (int r = 0; r < R; ++r) row_ok[r] = live && (l + P * r < n);
            T *Ac = A + l;
#pragma unroll
            for (int c = 0; c < N; ++c) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (P * r + P - 1 < c) continue;
                    const bool below = P * r >= c || l + P * r >= c;
                    if (row_ok[r] && below) Ac[P * r] = a[r][c];
                }
                Ac += lda;
            }
        } else {
            // U(c,i) = conj(L(i,c)): column i of U is row i of L; transpose through the slab,
            // one block of P rows (= P columns of U) at a time
#pragma unroll
            for (int cb = 0; cb < R; ++cb) {
                const int c0 = P * cb;
                if (c0 >= n) break;
                __syncwarp();
                const int i = c0 + l;
#pragma unroll
                for (int c = 0; c < P * cb + P; ++c)
                    if (c <= i) stage[l * LDU + c] = conj(a[cb][c]);
                __syncwarp();
                // U(r, colx) = conj(L(colx, r)) for r <= colx: column colx of U, rows by lane
                if (live) {
#pragma unroll
                    for (int ii = 0; ii < P; ++ii) {
                        const int colx = c0 + ii;
#pragma unroll
                        for (int t = 0; t <= cb; ++t) {
                            const int r = l + P * t;
                            if (colx < n && r <= colx) A[static_cast<int64_t>(colx) * lda + r] = stage[ii * LDU + r];
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
