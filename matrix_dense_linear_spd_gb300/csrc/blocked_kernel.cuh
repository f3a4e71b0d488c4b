// Blocked Cholesky family ("blocked"): one CTA per matrix, right-looking over panels of NB
// columns, the matrix updated in place in global memory (L2 holds the active matrices).
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "The blocked driver"): for
// j0 = 0, NB, 2NB, ...
//   1. factor the diagonal block L11 = chol(A11) (in shared memory);
//   2. panel solve L21 = A21 * L11^{-H} (one row per thread, L11 in shared memory);
//   3. trailing update A22 -= L21 * L21^H on the lower triangle only: tiles on or below the
//      diagonal, the diagonal tiles masked, so the other triangle is never written
//      ("The fold-free trailing update is ... wrong: it clobbers the upper triangle").
// A failure at local column c of a panel is reported at global column j0 + c + 1
// ("potrf: correctness findings" item 6), and the item stops there.
// Upper runs on the view S(i,k) = conj(A(k,i)); every global access is mapped so that the
// index that is contiguous in memory varies fastest across threads.
// posv / potrs: after the factor, forward (L*y = b, axpy form) and back (L^H*x = y, axpy form
// on the rows of L) substitution in global memory ("The fused potrs solve").
//
// Tensor-core variant (TC, f32 only): the trailing update -- the only dense contraction of the
// factorisation -- runs on the fifth-generation tensor cores. Each 128 x 128 lower tile of
// L21*L21^T is formed in tensor memory by tcgen05.mma kind::tf32 from 128-byte-swizzled
// K-major operand tiles in shared memory, with the 3xTF32 split (hi*hi + hi*lo + lo*hi, each
// f32 split into a rounded tf32 part and a tf32 remainder) so the product keeps f32 accuracy;
// the epilogue reads the tile back with tcgen05.ld and subtracts it from the lower triangle.
#pragma once

#include "bl_types.cuh"
#include "tc_sm100.cuh"

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

template <typename T, int NB, bool TC = false>
struct BlkCfg {
    static_assert(!TC || (NB <= 32 && sizeof(T) == 4), "tensor-core path: f32, panel width <= 32");
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
    // tensor-core path: the whole L21 panel stays resident as tf32 hi and lo operand panels
    // (TC_MAXM rows x 128 bytes each, 128-byte-swizzled K-major), next to the panel staging area
    static constexpr int TC_MAXM = 512;                        // trailing rows: n <= TC_MAXM + NB
    static constexpr size_t tc_panel = static_cast<size_t>(TC_MAXM) * 128;
    // epilogue staging: half a product tile (128 x 64 f32) with a padded row stride for Upper
    static constexpr int TC_STG_LD = 68;
    static constexpr size_t tc_stage = static_cast<size_t>(128) * TC_STG_LD * 4;
    static constexpr size_t tc_bytes = TC ? panel_bytes + 1024 + 2 * tc_panel + tc_stage : 0;
    static constexpr size_t simt_work = panel_bytes > trail_bytes ? panel_bytes : trail_bytes;
    static constexpr size_t work_bytes = simt_work > tc_bytes ? simt_work : tc_bytes;
    static constexpr size_t off_diag = 0;
    static constexpr size_t off_rs = off_diag + diag_bytes;
    static constexpr size_t off_work = ((off_rs + rs_bytes) + 15) / 16 * 16;
    static constexpr size_t smem_bytes = off_work + work_bytes;
};

template <typename T, int NB, bool TC = false>
__global__ void __launch_bounds__(256, TC ? 1 : 4) blocked_kernel(const BatchArgs args) {
    using C = BlkCfg<T, NB, TC>;
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
    // tensor-core resources: 128 tensor-memory columns (one 128 x 128 f32 tile) and an mbarrier
    __shared__ uint32_t s_tmem;
    __shared__ uint64_t s_mbar[2];
    uint32_t mma_phases = 0;                                   // bit b: parity of accumulator b
    if constexpr (TC) {
        if ((tid >> 5) == 0) {
            tc::tmem_alloc(&s_tmem, 256);                      // two 128 x 128 f32 accumulators
            tc::tmem_relinquish();
        }
        if (tid == 0) {
            tc::mbar_init(&s_mbar[0], 1);
            tc::mbar_init(&s_mbar[1], 1);
            tc::mbar_fence_init();
        }
        tc::fence_before_sync();
    }
    __syncthreads();
    if constexpr (TC) tc::fence_after_sync();

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
            if constexpr (TC) {
                // one warp factors the (<= 32) x 32 diagonal block in registers: lane r holds row
                // r; pivots and column entries travel by shuffles; the other warps wait
                __shared__ int s_diag_fail;
                if ((tid >> 5) == 0) {
                    const int lane = tid & 31;
                    float a[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) a[c] = (c <= lane && lane < kb) ? sD[c * LDD + lane] : (c == lane ? 1.f : 0.f);
                    unsigned failed = 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float d = __shfl_sync(0xffffffffu, a[j], j);
                        const bool ok = d > 0.f;
                        const float rs = ok ? rsqrtf(d) : 0.f;
                        failed |= (ok || j >= kb) ? 0u : (1u << j);
                        a[j] = (lane == j) ? (ok ? d * rs : d) : (lane > j ? a[j] * rs : a[j]);
#pragma unroll
                        for (int k = j + 1; k < 32; ++k) {
                            const float lk = __shfl_sync(0xffffffffu, a[j], k);
                            a[k] = fmaf(-a[j], lk, a[k]);
                        }
                        if (lane == j) sRs[j] = rs;
                    }
                    float *sL = reinterpret_cast<float *>(sW);        // L11 columns, stride 32
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (c <= lane && lane < kb) sD[c * LDD + lane] = a[c];
                        sL[c * 32 + lane] = (c < lane && lane < kb) ? a[c] : 0.f;
                    }
                    if (lane == 0) s_diag_fail = failed ? __ffs(failed) - 1 : -1;
                }
                __syncthreads();
                fail_col = s_diag_fail;
            } else
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
            const int mt_all = n - m0;
            unsigned char *p_hi = nullptr, *p_lo = nullptr;
            if constexpr (TC) {
                unsigned char *pb = reinterpret_cast<unsigned char *>(sW) + C::panel_bytes;
                pb += (1024 - (tc::smem_u32(pb) & 1023)) & 1023;
                p_hi = pb;
                p_lo = pb + C::tc_panel;
                // zero the padding rows of the last 128-row operand tile
                const int mpad = (mt_all + 127) / 128 * 128;
                for (int idx = tid; idx < (mpad - mt_all) * 32; idx += THREADS) {
                    const int row = mt_all + (idx >> 5), k = idx & 31;
                    const uint32_t off = tc::sw128_offset(row, k);
                    *reinterpret_cast<float *>(p_hi + off) = 0.f;
                    *reinterpret_cast<float *>(p_lo + off) = 0.f;
                }
            }
            if constexpr (TC) {
                // one row of A21 per thread, in registers: x_k = a_k / L(k,k), then
                // a_m -= x_k * L(m,k) for m > k (independent FMAs), L11 columns read as 16-byte
                // broadcasts; the solved row goes back to memory and, split into tf32 hi/lo, into
                // its row of the resident operand panels as 16-byte chunks
                const float *sL = reinterpret_cast<const float *>(sW);
                for (int rb = m0; rb < n; rb += THREADS) {
                    const int r = rb + tid;
                    if (r < n) {
                        float a[32];
#pragma unroll
                        for (int k = 0; k < 32; ++k) a[k] = re(S.get(r, j0 + k));
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const float x = a[k] * sRs[k];
                            a[k] = x;
#pragma unroll
                            for (int q = (k + 1) / 4; q < 8; ++q) {
                                const float4 l4 = *reinterpret_cast<const float4 *>(sL + k * 32 + 4 * q);
                                if (4 * q + 0 > k) a[4 * q + 0] = fmaf(-x, l4.x, a[4 * q + 0]);
                                if (4 * q + 1 > k) a[4 * q + 1] = fmaf(-x, l4.y, a[4 * q + 1]);
                                if (4 * q + 2 > k) a[4 * q + 2] = fmaf(-x, l4.z, a[4 * q + 2]);
                                if (4 * q + 3 > k) a[4 * q + 3] = fmaf(-x, l4.w, a[4 * q + 3]);
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 32; ++k) S.set(r, j0 + k, from_real<T>(a[k]));
                        const int prow = r - m0;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            float4 h4, l4;
                            tc::split_tf32(a[4 * q + 0], h4.x, l4.x);
                            tc::split_tf32(a[4 * q + 1], h4.y, l4.y);
                            tc::split_tf32(a[4 * q + 2], h4.z, l4.z);
                            tc::split_tf32(a[4 * q + 3], h4.w, l4.w);
                            const uint32_t off = tc::sw128_offset(prow, 4 * q);
                            *reinterpret_cast<float4 *>(p_hi + off) = h4;
                            *reinterpret_cast<float4 *>(p_lo + off) = l4;
                        }
                    }
                }
            } else
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
            if constexpr (TC) {
                // Every lower 128 x 128 tile (bi >= bk) of L21*L21^T, in a flat list. The
                // operands are rows of the resident panel; tile t accumulates in tensor-memory
                // buffer t&1, so the MMAs of tile t run while the epilogue of tile t-1 reads
                // buffer (t-1)&1 and subtracts it from the trailing matrix.
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncthreads();
                tc::fence_after_sync();
                const uint32_t tmem = s_tmem;
                const int warp = tid >> 5, lane = tid & 31;
                const int ntile = (mt + 127) / 128;
                const int T_all = ntile * (ntile + 1) / 2;
                const uint32_t s_hi = tc::smem_u32(p_hi), s_lo = tc::smem_u32(p_lo);
                int bi = 0, bk = 0;                  // tile t (issue side)
                int ei = 0, ek = 0;                  // tile t-1 (epilogue side)
                float *stg = reinterpret_cast<float *>(p_lo + C::tc_panel);
                // bulk adds need 16-byte aligned runs: lda a multiple of 4 and an aligned base
                const bool bulk_ok = (S.lda % 4 == 0) && ((reinterpret_cast<uintptr_t>(S.A) & 15) == 0);
                bool bulk_issued = false;            // issued since the last read-completion wait
                bool bulk_pending = false;           // issued since the last full-completion wait
                for (int t = 0; t <= T_all; ++t) {
                    if (t < T_all && tid == 0) {
                        constexpr uint32_t idesc = tc::idesc_tf32(128, 128);
                        const uint32_t d = tmem + static_cast<uint32_t>((t & 1) * 128);
                        const uint32_t a_hi = s_hi + bi * 16384, a_lo = s_lo + bi * 16384;
                        const uint32_t b_hi = s_hi + bk * 16384, b_lo = s_lo + bk * 16384;
                        for (int st = 0; st < 4; ++st)
                            tc::mma_tf32(d, tc::sdesc_sw128(a_hi + 32 * st), tc::sdesc_sw128(b_hi + 32 * st), idesc, st > 0);
                        for (int st = 0; st < 4; ++st)
                            tc::mma_tf32(d, tc::sdesc_sw128(a_hi + 32 * st), tc::sdesc_sw128(b_lo + 32 * st), idesc, true);
                        for (int st = 0; st < 4; ++st)
                            tc::mma_tf32(d, tc::sdesc_sw128(a_lo + 32 * st), tc::sdesc_sw128(b_hi + 32 * st), idesc, true);
                        tc::mma_commit(&s_mbar[t & 1]);
                    }
                    if (t >= 1) {
                        const int u = t - 1, buf = u & 1;
                        const bool done = tc::mbar_wait(&s_mbar[buf], (mma_phases >> buf) & 1u, 1u << 22);
                        mma_phases ^= 1u << buf;
                        tc::fence_after_sync();
                        if (!done) {
                            if (tid == 0) { args.info[mat] = -1; s_fail = 1; }
                        } else {
                            // Epilogue, half a tile (64 columns) at a time: TMEM -> registers ->
                            // staging (negated) -> asynchronous bulk adds into the trailing matrix,
                            // one contiguous run per column (Lower) or per row of S (Upper). Runs
                            // that do not start on a 16-byte boundary are done element-wise.
                            const int row = 32 * (warp & 3) + lane;
                            const int I0 = m0 + ei * 128, K0 = m0 + ek * 128;
                            for (int h = 0; h < 2; ++h) {
                                if (bulk_issued) { tc::bulk_wait_read_all(); bulk_issued = false; }
                                __syncthreads();
                                const int cl0 = 32 * (warp >> 2);            // column inside the half
                                float v[32];
                                tc::tmem_ld32(tmem + static_cast<uint32_t>(buf * 128) +
                                                  (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 64 * h + cl0,
                                              v);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    if (!upper) stg[(cl0 + i) * 128 + row] = -v[i];
                                    else stg[row * C::TC_STG_LD + cl0 + i] = -v[i];
                                }
                                tc::fence_proxy_async_smem();
                                __syncthreads();
                                if (!upper) {
                                    if (tid < 64) {
                                        const int gk = K0 + 64 * h + tid;
                                        const int lo = max(I0, gk), hi = min(I0 + 128, n);
                                        if (gk < n && lo < hi) {
                                            float *colp = S.A + static_cast<int64_t>(gk) * S.lda;
                                            const float *src = stg + tid * 128 - I0;
                                            int la = lo, ha = lo;
                                            if (bulk_ok) {
                                                la = min((lo + 3) & ~3, hi);
                                                ha = max(la, hi & ~3);
                                            }
                                            for (int gi = lo; gi < la; ++gi) colp[gi] += src[gi];
                                            if (ha > la) {
                                                tc::bulk_reduce_add_f32(colp + la, src + la, static_cast<uint32_t>((ha - la) * 4));
                                                bulk_issued = bulk_pending = true;
                                            }
                                            for (int gi = max(ha, la); gi < hi; ++gi) colp[gi] += src[gi];
                                        }
                                    }
                                } else {
                                    if (tid < 128) {
                                        const int gi = I0 + tid;
                                        const int lo = K0 + 64 * h, hi = min(min(lo + 64, gi + 1), n);
                                        if (gi < n && lo < hi) {
                                            float *rowp = S.A + static_cast<int64_t>(gi) * S.lda;
                                            const float *src = stg + tid * C::TC_STG_LD - lo;
                                            int ha = lo;
                                            if (bulk_ok) ha = lo + ((hi - lo) & ~3);
                                            if (ha > lo) {
                                                tc::bulk_reduce_add_f32(rowp + lo, src + lo, static_cast<uint32_t>((ha - lo) * 4));
                                                bulk_issued = bulk_pending = true;
                                            }
                                            for (int gk = ha; gk < hi; ++gk) rowp[gk] += src[gk];
                                        }
                                    }
                                }
                                if (bulk_issued) tc::bulk_commit();
                            }
                        }
                        tc::fence_before_sync();
                        ei = bi;
                        ek = bk;
                    } else {
                        ei = bi;
                        ek = bk;
                    }
                    // advance the issue-side tile
                    if (++bk > bi) { ++bi; bk = 0; }
                    __syncthreads();
                    tc::fence_after_sync();
                }
                // the bulk adds must have landed before anyone reads the trailing matrix again
                if (bulk_pending) tc::bulk_wait_all();
                tc::fence_proxy_async_all();
                __syncthreads();
                if (s_fail) break;
                continue;
            }
            const int ntile = (mt + TB - 1) / TB;
            T *sI = sW;
            T *sK = sW + NB * LDT;
            const int ti = upper ? tid / 16 : tid % 16;   // row group (4 rows)
            const int tk = upper ? tid % 16 : tid / 16;   // column group (4 columns)
            for (int bi = 0; bi < ntile; ++bi) {
                const int I0 = m0 + bi * TB;
                for (int bk = 0; bk <= bi; ++bk) {
                    const int K0 = m0 + bk * TB;
                    for (int idx = tid; idx < kb * TB; idx += THREADS) {
                        const int a0 = upper ? idx % kb : idx % TB;
                        const int a1 = upper ? idx / kb : idx / TB;
                        const int rr = upper ? a1 : a0, c = upper ? a0 : a1;
                        sI[c * LDT + rr] = (I0 + rr < n) ? S.get(I0 + rr, j0 + c) : zero<T>();
                        sK[c * LDT + rr] = (K0 + rr < n) ? S.get(K0 + rr, j0 + c) : zero<T>();
                    }
                    __syncthreads();
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
                    __syncthreads();
                }
            }
        }
        if (tid == 0 && !s_fail) args.info[mat] = 0;
        __syncthreads();
    }
    if constexpr (TC) {
        tc::fence_before_sync();
        __syncthreads();
        if ((tid >> 5) == 0) tc::tmem_dealloc(s_tmem, 256);
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
