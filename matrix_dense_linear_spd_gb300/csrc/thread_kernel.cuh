// Thread-per-matrix Cholesky family ("thread"): each thread factors one whole matrix, held as a
// packed triangle in shared memory, for small n.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page: the factor A = L*L^H, info = first
// non-positive pivot, Upper as a load/store transform): Cholesky-Banachiewicz, row by row --
//   L(i,j) = (A(i,j) - sum_{k<j} L(i,k) * conj(L(j,k))) / L(j,j),  j < i,
//   d = Re A(i,i) - sum_{k<i} |L(i,k)|^2;  stop with info = i+1 if !(d > 0), else L(i,i) = sqrt(d).
// Upper runs the same recurrence on S(i,j) = conj(A(j,i)); the conjugation is applied where each
// input value is first read, so the copy into shared memory is a plain byte copy.
//
// Why a thread per matrix: GB300 executes FP64 at 2 lanes per clock per SM, 1/64 of its FP32
// rate, so every f64 cell is bound by FP64 instructions issued, and any layout that spreads
// one small matrix over many lanes (predicated-off or padded lanes still occupy the FP64 pipe)
// wastes most of it. Here every lane of every FP64 instruction does useful work, and a few warps
// per SM keep the FP64 pipe busy (a warp-wide FP64 instruction holds it for 16 clocks).
//
// Data movement: the CTA's triangles arrive by asynchronous element copies (cp.async, no
// register round trip, all in flight at once) in global-address order, so a warp's copies are
// coalesced; a per-CTA table maps each position of an n x n item to its packed slot, so the
// copy loop needs no division, and for items stored back to back the global offset is the flat
// index itself. The per-matrix stride keeps the factorisation's shared-memory accesses
// bank-conflict free (see ThreadCfg).
//
// Variants: a pair of lanes per matrix (TPMX = 2), each lane summing one parity of every dot
// product; and the one-lane factor fully unrolled at n == NMAX (EXACT). Both perform the row
// loop's operations in the row loop's order, so all variants give the same bits.
#pragma once

#include "bl_types.cuh"

namespace bl {

// TPMX threads per matrix: 1, or 2 (a pair of adjacent lanes splits every dot product by the
// parity of its index k; see the kernel).
template <typename T, int NMAX, int TPMX = 1>
struct ThreadCfg {
    static constexpr int TRI = NMAX * (NMAX + 1) / 2;            // packed lower triangle, row-major
    static constexpr int rsw = (NMAX * static_cast<int>(sizeof(real_t<T>)) + static_cast<int>(sizeof(T)) - 1) /
                               static_cast<int>(sizeof(T));
    static constexpr int PACK0 = TRI + rsw;                      // packed triangle + NMAX reciprocal pivots
    // per-matrix stride in elements. One thread per matrix: odd in 8-byte words, so the 16 lanes of
    // a half-warp (16 matrices, same offset) hit distinct banks. Two: a half-warp phase is 8
    // matrices x 2 lanes at offsets c and c+1, distinct banks when the stride is 2 modulo the
    // phase's width in elements (16 for 8-byte, 8 for 16-byte elements).
    static constexpr int pack_stride() {
        if (TPMX == 1) return (((PACK0 * static_cast<int>(sizeof(T))) / 8) % 2) ? PACK0 : PACK0 + 1;
        const int w = sizeof(T) >= 16 ? 8 : 16;
        int p = PACK0;
        while (p % w != 2) ++p;
        return p;
    }
    static constexpr int PACK = pack_stride();
    static constexpr size_t table_bytes = sizeof(uint32_t) * NMAX * NMAX;
    static constexpr size_t bytes_for(int mats) { return sizeof(T) * static_cast<size_t>(PACK) * mats + table_bytes; }
    // one thread per matrix: as many matrices per CTA as fit one CTA's shared memory, up to 128;
    // two: 64 matrices (128 threads) per CTA, so two CTAs share an SM where the first holds one
    static constexpr int THREADS = TPMX == 1 ? (bytes_for(128) <= 227 * 1024 ? 128 : 64)
                                             : (bytes_for(64) <= 227 * 1024 ? 128 : 64);
    static constexpr int MATS = THREADS / TPMX;                  // matrices per CTA
    static constexpr size_t smem_bytes = bytes_for(MATS);
};

__device__ __forceinline__ int tri_idx(int i, int j) { return i * (i + 1) / 2 + j; }

// One matrix per thread at the compile-time order N: the one-thread kernel's row loop (below)
// with every loop unrolled, so every shared-memory offset is an immediate, no loop control is
// left and the compiler may keep row i in registers; the operations and their order are the
// row loop's, so the results are bit-identical to it. Returns info.
template <typename T, int N>
__device__ __forceinline__ int factor_exact(T *a, bool upper) {
    using R = real_t<T>;
    R *rinv = reinterpret_cast<R *>(a + N * (N + 1) / 2);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        T *ri = a + tri_idx(i, 0);
#pragma unroll
        for (int j = 0; j + 1 < i; j += 2) {
            const T *rj = a + tri_idx(j, 0);
            const T *rj1 = rj + j + 1;
            T sa0 = upper ? conj(ri[j]) : ri[j], sb0 = upper ? conj(ri[j + 1]) : ri[j + 1];
            T sa1 = zero<T>(), sb1 = zero<T>();
#pragma unroll
            for (int k = 0; k + 1 < j; k += 2) {
                const T x0 = ri[k], x1 = ri[k + 1];
                sub_mul_conj(sa0, x0, rj[k]);
                sub_mul_conj(sb0, x0, rj1[k]);
                sub_mul_conj(sa1, x1, rj[k + 1]);
                sub_mul_conj(sb1, x1, rj1[k + 1]);
            }
            add_into(sa0, sa1);                                  // j even: no odd leftover k
            add_into(sb0, sb1);
            const T lij = scale(sa0, rinv[j]);
            ri[j] = lij;
            sub_mul_conj(sb0, lij, rj1[j]);
            ri[j + 1] = scale(sb0, rinv[j + 1]);
        }
        if (i & 1) {                                             // leftover entry j = i-1 (even)
            const int j = i - 1;
            const T *rj = a + tri_idx(j, 0);
            T s0 = upper ? conj(ri[j]) : ri[j], s1 = zero<T>();
#pragma unroll
            for (int k = 0; k + 1 < j; k += 2) {
                sub_mul_conj(s0, ri[k], rj[k]);
                sub_mul_conj(s1, ri[k + 1], rj[k + 1]);
            }
            add_into(s0, s1);
            ri[j] = scale(s0, rinv[j]);
        }
        R d0 = re(ri[i]), d1 = R(0), d2 = R(0), d3 = R(0);
#pragma unroll
        for (int k = 0; k + 3 < i; k += 4) {
            sub_abs2(d0, ri[k]);
            sub_abs2(d1, ri[k + 1]);
            sub_abs2(d2, ri[k + 2]);
            sub_abs2(d3, ri[k + 3]);
        }
#pragma unroll
        for (int k = (i / 4) * 4; k < i; ++k) sub_abs2(d0, ri[k]);
        const R dd = (d0 + d1) + (d2 + d3);
        if (!(dd > R(0))) return i + 1;
        const R r = rsqrt_of(dd);
        ri[i] = from_real<T>(dd * r);
        rinv[i] = r;
    }
    return 0;
}

// The value of the other lane of an adjacent-lane pair (mask m names the pair's two lanes).
__device__ __forceinline__ double shfl_xor_pair(double v, unsigned m) { return __shfl_xor_sync(m, v, 1); }
__device__ __forceinline__ cf64 shfl_xor_pair(cf64 v, unsigned m) {
    return cf64{__shfl_xor_sync(m, v.x, 1), __shfl_xor_sync(m, v.y, 1)};
}

// EXACT: when n == NMAX the one-thread factor runs fully unrolled (factor_exact); other orders
// run the row loop.
template <typename T, int NMAX, int TPMX = 1, bool EXACT = false>
__global__ void __launch_bounds__(ThreadCfg<T, NMAX, TPMX>::THREADS, 1) thread_kernel(const BatchArgs args) {
    using C = ThreadCfg<T, NMAX, TPMX>;
    using R = real_t<T>;
    constexpr int THREADS = C::THREADS, PACK = C::PACK, TRI = C::TRI, MATS = C::MATS;
    extern __shared__ __align__(16) unsigned char smem[];
    T *sm = reinterpret_cast<T *>(smem);
    uint32_t *tab = reinterpret_cast<uint32_t *>(smem + sizeof(T) * static_cast<size_t>(PACK) * MATS);

    const int tid = threadIdx.x;
    const int n = args.n;
    const bool upper = args.upper != 0;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * MATS;
    const int nm = static_cast<int>(args.batch - m0 < MATS ? args.batch - m0 : MATS);   // live matrices
    const int64_t lda = args.lda, sa = args.stride_a;
    const int nn = n * n;

    // position rem = col * n + row of the n x n item -> bits 0-15 its packed slot (0xFFFF: not
    // referenced), bits 16-23 col, bits 24-31 row
    for (int rem = tid; rem < nn; rem += THREADS) {
        const int col = rem / n, row = rem - col * n;
        const bool ref = upper ? row <= col : row >= col;
        const uint32_t slot = ref ? static_cast<uint32_t>(upper ? tri_idx(col, row) : tri_idx(row, col)) : 0xFFFFu;
        tab[rem] = slot | (static_cast<uint32_t>(col) << 16) | (static_cast<uint32_t>(row) << 24);
    }
    __syncthreads();

    // flat index idx = mm * nn + rem over the CTA's items, walked in steps of THREADS without division
    const int dm = THREADS / nn, dr = THREADS - (THREADS / nn) * nn;
    const T *A = static_cast<const T *>(args.A) + m0 * sa;
    // items stored back to back (lda = n, stride = n^2): the global offset is the flat index
    // itself, so the walk needs no 64-bit index arithmetic per element
    const bool flat = lda == n && sa == nn;
    if (flat) {
        int mb = (tid / nn) * PACK, rem = tid - (tid / nn) * nn;
        for (int idx = tid; idx < nm * nn; idx += THREADS) {
            const uint32_t slot = tab[rem] & 0xFFFFu;
            if (slot != 0xFFFFu) cp_async_elem<sizeof(T)>(sm + mb + slot, A + idx);
            mb += dm * PACK;
            rem += dr;
            if (rem >= nn) rem -= nn, mb += PACK;
        }
    } else {
        int mm = tid / nn, rem = tid - (tid / nn) * nn;
        for (int idx = tid; idx < nm * nn; idx += THREADS) {
            const uint32_t e = tab[rem];
            const uint32_t slot = e & 0xFFFFu;
            if (slot != 0xFFFFu) {
                const int col = (e >> 16) & 0xFF, row = e >> 24;
                cp_async_elem<sizeof(T)>(sm + mm * PACK + slot, A + mm * sa + col * lda + row);
            }
            mm += dm;
            rem += dr;
            if (rem >= nn) rem -= nn, ++mm;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    int info = 0;
    if constexpr (TPMX == 1) {
        // ---- one matrix per thread. Two entries of row i at a time (j, j+1): the shared loads of
        // L(i,k) feed both dot products, and each is split in two partial sums, so four independent
        // FP64 chains are in flight per thread (the FP64 pipe's latency is long).
        bool done = false;
        if constexpr (EXACT) {
            if (tid < nm && n == NMAX) {
                info = factor_exact<T, NMAX>(sm + tid * PACK, upper);
                done = true;
            }
        }
        if (tid < nm && !done) {
            T *a = sm + tid * PACK;
            R *rinv = reinterpret_cast<R *>(a + TRI);
            for (int i = 0; i < n; ++i) {
                T *ri = a + tri_idx(i, 0);
                int j = 0;
                for (; j + 1 < i; j += 2) {
                    const T *rj = a + tri_idx(j, 0);
                    const T *rj1 = rj + j + 1;                    // row j+1 follows row j
                    T sa0 = upper ? conj(ri[j]) : ri[j], sb0 = upper ? conj(ri[j + 1]) : ri[j + 1];
                    T sa1 = zero<T>(), sb1 = zero<T>();
                    int k = 0;
                    for (; k + 1 < j; k += 2) {
                        const T x0 = ri[k], x1 = ri[k + 1];
                        sub_mul_conj(sa0, x0, rj[k]);
                        sub_mul_conj(sb0, x0, rj1[k]);
                        sub_mul_conj(sa1, x1, rj[k + 1]);
                        sub_mul_conj(sb1, x1, rj1[k + 1]);
                    }
                    if (k < j) {
                        const T x0 = ri[k];
                        sub_mul_conj(sa0, x0, rj[k]);
                        sub_mul_conj(sb0, x0, rj1[k]);
                    }
                    add_into(sa0, sa1);
                    add_into(sb0, sb1);
                    const T lij = scale(sa0, rinv[j]);
                    ri[j] = lij;
                    sub_mul_conj(sb0, lij, rj1[j]);
                    ri[j + 1] = scale(sb0, rinv[j + 1]);
                }
                if (j < i) {                                      // odd leftover entry j = i-1
                    const T *rj = a + tri_idx(j, 0);
                    T s0 = upper ? conj(ri[j]) : ri[j], s1 = zero<T>();
                    int k = 0;
                    for (; k + 1 < j; k += 2) {
                        sub_mul_conj(s0, ri[k], rj[k]);
                        sub_mul_conj(s1, ri[k + 1], rj[k + 1]);
                    }
                    if (k < j) sub_mul_conj(s0, ri[k], rj[k]);
                    add_into(s0, s1);
                    ri[j] = scale(s0, rinv[j]);
                }
                R d0 = re(ri[i]), d1 = R(0), d2 = R(0), d3 = R(0);
                int k = 0;
                for (; k + 3 < i; k += 4) {
                    sub_abs2(d0, ri[k]);
                    sub_abs2(d1, ri[k + 1]);
                    sub_abs2(d2, ri[k + 2]);
                    sub_abs2(d3, ri[k + 3]);
                }
                for (; k < i; ++k) sub_abs2(d0, ri[k]);
                const R dd = (d0 + d1) + (d2 + d3);
                if (!(dd > R(0))) {
                    info = i + 1;
                    break;
                }
                const R r = rsqrt_of(dd);
                ri[i] = from_real<T>(dd * r);
                rinv[i] = r;
            }
        }
    } else {
        // ---- a pair of adjacent lanes per matrix. Lane h of the pair runs the chains of the
        // one-thread kernel that sum over k = h (mod 2) -- the even chains start from A(i,j),
        // the odd ones from zero, exactly as there -- and the pair adds them with one shuffle in
        // the same order, so every entry is bit-identical to the one-thread kernel's. Lane h keeps
        // the row entries of its parity (its later dot products read only those, plus L(j+1,j)
        // of an earlier row); lane 0 also keeps the diagonal and the reciprocal pivots, and the
        // pair syncs once per row. A pair that stops at a failed pivot stops together (both
        // lanes hold the same pivot), and shuffles and syncs name only the pair's two lanes.
        const int mloc = tid >> 1, h = tid & 1;
        const unsigned pm = 3u << ((tid & 31) & ~1);
        if (mloc < nm) {
            T *a = sm + mloc * PACK;
            R *rinv = reinterpret_cast<R *>(a + TRI);
            for (int i = 0; i < n; ++i) {
                T *ri = a + tri_idx(i, 0);
                int j = 0;
                for (; j + 1 < i; j += 2) {
                    const T *rj = a + tri_idx(j, 0);
                    const T *rj1 = rj + j + 1;
                    T sa = zero<T>(), sb = zero<T>();
                    if (h == 0) {
                        sa = upper ? conj(ri[j]) : ri[j];
                        sb = upper ? conj(ri[j + 1]) : ri[j + 1];
                    }
                    int k = h;
                    for (; k < j; k += 2) {
                        const T x = ri[k];
                        sub_mul_conj(sa, x, rj[k]);
                        sub_mul_conj(sb, x, rj1[k]);
                    }
                    const T sa_o = shfl_xor_pair(sa, pm), sb_o = shfl_xor_pair(sb, pm);
                    T ta = h == 0 ? sa : sa_o, tb = h == 0 ? sb : sb_o;       // the even chains
                    add_into(ta, h == 0 ? sa_o : sa);                         // + the odd chains
                    add_into(tb, h == 0 ? sb_o : sb);
                    const T lij = scale(ta, rinv[j]);
                    sub_mul_conj(tb, lij, rj1[j]);
                    const T lij1 = scale(tb, rinv[j + 1]);
                    if (h == 0) ri[j] = lij;
                    else ri[j + 1] = lij1;
                }
                if (j < i) {                                  // odd leftover entry j = i-1 (even)
                    const T *rj = a + tri_idx(j, 0);
                    T sv = (h == 0) ? (upper ? conj(ri[j]) : ri[j]) : zero<T>();
                    for (int k = h; k < j; k += 2) sub_mul_conj(sv, ri[k], rj[k]);
                    const T so = shfl_xor_pair(sv, pm);
                    T t0 = h == 0 ? sv : so;
                    add_into(t0, h == 0 ? so : sv);
                    if (h == 0) ri[j] = scale(t0, rinv[j]);
                }
                // the diagonal: the one-thread kernel's four chains over k mod 4 (lane h holds
                // chains h and h + 2), the entries past the last whole group of four all in chain 0
                __syncwarp(pm);                               // both parities of row i are stored
                R dA = (h == 0) ? re(ri[i]) : R(0), dB = R(0);
                int k = 0;
                for (; k + 3 < i; k += 4) {
                    sub_abs2(dA, ri[k + h]);
                    sub_abs2(dB, ri[k + 2 + h]);
                }
                if (h == 0)
                    for (; k < i; ++k) sub_abs2(dA, ri[k]);
                const R dA_o = __shfl_xor_sync(pm, dA, 1), dB_o = __shfl_xor_sync(pm, dB, 1);
                const R x01 = h == 0 ? dA + dA_o : dA_o + dA;   // d0 + d1
                const R x23 = h == 0 ? dB + dB_o : dB_o + dB;   // d2 + d3
                const R dd = x01 + x23;
                if (!(dd > R(0))) {
                    info = i + 1;
                    break;
                }
                const R r = rsqrt_of(dd);
                if (h == 0) {
                    ri[i] = from_real<T>(dd * r);
                    rinv[i] = r;
                }
                __syncwarp(pm);                               // the row is complete for both lanes
            }
        }
    }
    __syncthreads();

    // ---- store of the referenced triangles, same walk (coalesced global writes)
    T *Aw = static_cast<T *>(args.A) + m0 * sa;
    if (flat) {
        int mb = (tid / nn) * PACK, rem = tid - (tid / nn) * nn;
        for (int idx = tid; idx < nm * nn; idx += THREADS) {
            const uint32_t slot = tab[rem] & 0xFFFFu;
            if (slot != 0xFFFFu) {
                const T v = sm[mb + slot];
                Aw[idx] = upper ? conj(v) : v;
            }
            mb += dm * PACK;
            rem += dr;
            if (rem >= nn) rem -= nn, mb += PACK;
        }
    } else {
        int mm = tid / nn, rem = tid - (tid / nn) * nn;
        for (int idx = tid; idx < nm * nn; idx += THREADS) {
            const uint32_t e = tab[rem];
            const uint32_t slot = e & 0xFFFFu;
            if (slot != 0xFFFFu) {
                const int col = (e >> 16) & 0xFF, row = e >> 24;
                const T v = sm[mm * PACK + slot];
                Aw[mm * sa + col * lda + row] = upper ? conj(v) : v;
            }
            mm += dm;
            rem += dr;
            if (rem >= nn) rem -= nn, ++mm;
        }
    }
    if (TPMX == 1 && tid < nm) args.info[m0 + tid] = info;
    if (TPMX == 2 && (tid & 1) == 0 && (tid >> 1) < nm) args.info[m0 + (tid >> 1)] = info;
}

}  // namespace bl
