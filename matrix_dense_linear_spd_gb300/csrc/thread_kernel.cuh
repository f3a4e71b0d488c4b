// Thread-per-matrix Cholesky family ("thread"): each thread factors one whole matrix, held as a
// packed triangle in shared memory, for small n.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page: the factor A = L*L^H, info = first
// non-positive pivot, Upper as a load/store transform): Cholesky-Banachiewicz, row by row --
//   L(i,j) = (A(i,j) - sum_{k<j} L(i,k) * conj(L(j,k))) / L(j,j),  j < i,
//   d = Re A(i,i) - sum_{k<i} |L(i,k)|^2;  stop with info = i+1 if !(d > 0), else L(i,i) = sqrt(d).
//
// Why a thread per matrix: GB300 executes FP64 at 2 lanes per clock per SM, 1/64 of its FP32
// rate, so every f64 cell is bound by FP64 instructions issued, and any layout that spreads
// one small matrix over many lanes (predicated-off or padded lanes still occupy the FP64 pipe)
// wastes most of it. Here every lane of every FP64 instruction does useful work. One warp per
// SM sub-partition keeps the FP64 units busy: a warp-wide FP64 instruction occupies its unit
// for 16 clocks, far longer than any dependency latency. Loads and stores are cooperative and
// coalesced (the CTA's matrices are one contiguous range in the common layout); the packed
// stride is odd in 8-byte words so per-thread accesses are bank-conflict free.
#pragma once

#include "bl_types.cuh"

namespace bl {

template <typename T, int NMAX>
struct ThreadCfg {
    static constexpr int THREADS = 128;
    static constexpr int TRI = NMAX * (NMAX + 1) / 2;            // packed lower triangle, row-major
    static constexpr int WORDS = static_cast<int>(sizeof(T) / 4);
    // packed triangle + NMAX reciprocal pivots; stride odd in 8-byte units (conflict-free)
    static constexpr int rsw = (NMAX * static_cast<int>(sizeof(real_t<T>)) + static_cast<int>(sizeof(T)) - 1) /
                               static_cast<int>(sizeof(T));
    static constexpr int PACK0 = TRI + rsw;
    static constexpr int PACK = (((PACK0 * static_cast<int>(sizeof(T))) / 8) % 2) ? PACK0 : PACK0 + 1;
    static constexpr size_t smem_bytes = sizeof(T) * static_cast<size_t>(PACK) * THREADS;
};

__device__ __forceinline__ int tri_idx(int i, int j) { return i * (i + 1) / 2 + j; }

template <typename T, int NMAX>
__global__ void __launch_bounds__(128, 1) thread_kernel(const BatchArgs args) {
    using C = ThreadCfg<T, NMAX>;
    using R = real_t<T>;
    constexpr int THREADS = C::THREADS, PACK = C::PACK, TRI = C::TRI;
    extern __shared__ __align__(16) unsigned char smem[];
    T *sm = reinterpret_cast<T *>(smem);

    const int tid = threadIdx.x;
    const int n = args.n;
    const bool upper = args.upper != 0;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * THREADS;
    const int nm = static_cast<int>(args.batch - m0 < THREADS ? args.batch - m0 : THREADS);   // live matrices
    const T *A = static_cast<const T *>(args.A);
    const int64_t lda = args.lda, sa = args.stride_a;
    const int nn = n * n;

    // ---- cooperative load of the referenced triangles (contiguous index fastest)
    for (int idx = tid; idx < nm * nn; idx += THREADS) {
        const int mm = idx / nn, rem = idx - mm * nn;
        const int col = rem / n, row = rem - col * n;                 // A(row, col)
        const T v = A[(m0 + mm) * sa + static_cast<int64_t>(col) * lda + row];
        if (!upper) {
            if (row >= col) sm[mm * PACK + tri_idx(row, col)] = v;
        } else {
            if (row <= col) sm[mm * PACK + tri_idx(col, row)] = conj(v);   // S(col,row) = conj(A(row,col))
        }
    }
    __syncthreads();

    // ---- one matrix per thread
    int info = 0;
    if (tid < nm) {
        T *a = sm + tid * PACK;
        R *rinv = reinterpret_cast<R *>(a + TRI);
        for (int i = 0; i < n; ++i) {
            T *ri = a + tri_idx(i, 0);
            for (int j = 0; j < i; ++j) {
                const T *rj = a + tri_idx(j, 0);
                T s = ri[j];
                for (int k = 0; k < j; ++k) sub_mul_conj(s, ri[k], rj[k]);
                ri[j] = scale(s, rinv[j]);
            }
            R d = re(ri[i]);
            for (int k = 0; k < i; ++k) {
                const T v = ri[k];
                d -= re(v) * re(v) + (is_cplx<T>::value ? im_part(v) * im_part(v) : R(0));
            }
            if (!(d > R(0))) {
                info = i + 1;
                break;
            }
            const R r = rsqrt_of(d);
            ri[i] = from_real<T>(d * r);
            rinv[i] = r;
        }
    }
    __syncthreads();

    // ---- cooperative store of the referenced triangles
    T *Aw = static_cast<T *>(args.A);
    for (int idx = tid; idx < nm * nn; idx += THREADS) {
        const int mm = idx / nn, rem = idx - mm * nn;
        const int col = rem / n, row = rem - col * n;
        if (!upper) {
            if (row >= col) Aw[(m0 + mm) * sa + static_cast<int64_t>(col) * lda + row] = sm[mm * PACK + tri_idx(row, col)];
        } else {
            if (row <= col) Aw[(m0 + mm) * sa + static_cast<int64_t>(col) * lda + row] = conj(sm[mm * PACK + tri_idx(col, row)]);
        }
    }
    if (tid < nm) args.info[m0 + tid] = info;
}

}  // namespace bl
