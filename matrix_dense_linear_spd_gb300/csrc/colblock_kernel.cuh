// Column-block tensor-core Cholesky ("blocked:nb=32:tc=2"), f32, n <= 512: one CTA per matrix,
// the current block of 128 columns held as f32 accumulators in tensor memory.
//
// Method (BatchLAS "Batched Cholesky (potrf)" page, section "The blocked driver": factor the
// diagonal block, solve the panel below it, update the rest; the update is the only dense
// contraction). The columns are taken in blocks of W = 128; for the block C0 .. C0+W-1, whose
// lower part has M = n - C0 rows:
//   1. block update on the tensor cores, left-looking: D = L(C0:n, 0:C0) * L(C0:C0+W, 0:C0)^T,
//      K in chunks of 32 columns of L. Each chunk is read once from global memory (two chunks
//      ahead, into registers), split into tf32 hi and lo parts (3xTF32: hi*hi + hi*lo + lo*hi
//      keeps f32 accuracy) and stored as a 128-byte-swizzled K-major operand panel (two panels,
//      alternating, so a chunk is staged while the previous one multiplies); the B operand is
//      the panel's first W rows. D lives in tensor memory, one 128 x W tile per 128 rows (4 tiles
//      = all 512 columns).
//   2. the block column is factored right-looking, 32 columns (one slice) at a time. The slice's
//      current values V = S(:, slice) - D(:, slice) are the original values from global memory
//      minus the accumulator read back with tcgen05.ld. One warp factors the 32 x 32 diagonal
//      block (first non-positive pivot fails the item) and inverts it; meanwhile the other rows
//      go, split, into the operand panel. The panel solve L21 = V * L11^-T then runs on the
//      tensor cores as V * Linv^T into the slice's own accumulator columns; the rows are read
//      back, written to global memory and, when the block has further slices, split into the
//      panel again, from where the tensor cores add L21 * L21^T to D for the block's remaining
//      columns.
// Each element of the referenced triangle is read from global memory once as input and written
// once; later blocks read finished L columns (from L2) as operands. Using L11^-1 for the panel
// solve adds a relative error of order cond(L11) * eps (cond(L11) <= sqrt(cond(A))).
//
// Upper runs on the view S(i,k) = A(k,i) (real type: no conjugation); only the referenced
// triangle is ever written. A failure at column c reports info = c + 1 and the item stops (the
// columns before c are final). Every wait on the tensor cores is bounded; a wait that gives up
// reports info = -1.
#pragma once

#include "bl_types.cuh"
#include "tc_sm100.cuh"

namespace bl {

struct ColBlkCfg {
    static constexpr int THREADS = 256;
    static constexpr int W = 128;                                   // block width (accumulator columns)
    static constexpr int MAXN = 512;                                // 4 row tiles x 128 tensor-memory columns
    // operand panels: rows x 32 tf32 (128 bytes), hi and lo parts. Panel 0 holds up to MAXN rows
    // (the slices of the first block); panel 1, the second buffer of the block update, up to
    // MAXN - W rows (blocks after the first). The diagonal block's L columns, its reciprocal
    // pivots and its inverse (the B tile of the panel solve) live in panel 1's space: the slices
    // never use panel 1, and no block-update MMA is in flight while a slice runs.
    static constexpr size_t P0_HI = 0;
    static constexpr size_t P0_LO = static_cast<size_t>(MAXN) * 128;
    static constexpr size_t P1_HI = 2 * P0_LO;
    static constexpr size_t P1_LO = P1_HI + static_cast<size_t>(MAXN - W) * 128;
    static constexpr size_t OFF_L11 = P1_HI;                        // sLs[c*32 + m] = L(c+m, c)
    static constexpr size_t OFF_RS = OFF_L11 + 32 * 32 * 4;         // 1 / L(c, c)
    static constexpr size_t OFF_BI_HI = P1_HI + 8192;               // Linv, 32 rows x 128 bytes, hi
    static constexpr size_t OFF_BI_LO = OFF_BI_HI + 4096;           // and lo
    static constexpr size_t END = P1_LO + static_cast<size_t>(MAXN - W) * 128;
    static constexpr size_t smem_bytes = 1024 + END;                // + 1024 for the panel alignment
    static_assert(OFF_RS + 32 * 4 <= OFF_BI_HI && OFF_BI_LO + 4096 <= END, "diagonal-block area inside panel 1");
};

namespace colblk {

// Offset of S(i, k) in the stored matrix: Lower S = A, Upper S(i,k) = A(k,i).
template <bool UPPER>
__device__ __forceinline__ int64_t sidx(int i, int k, int64_t lda) {
    return UPPER ? static_cast<int64_t>(i) * lda + k : static_cast<int64_t>(k) * lda + i;
}

// S(i, k0 + c) for c < 32 into v; entries with k0 + c >= kend are 0 (kend <= k0: all 0). Upper
// rows of S are contiguous in memory: with `vec` (16-byte aligned rows) a whole row moves as
// eight 16-byte loads instead of 32 scattered ones.
template <bool UPPER>
__device__ __forceinline__ void load_row(const float *A, int64_t lda, int i, int k0, int kend, float (&v)[32],
                                         bool vec) {
    if (UPPER && vec && kend >= k0 + 32) {
        const float4 *p = reinterpret_cast<const float4 *>(A + static_cast<int64_t>(i) * lda + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 t = p[q];
            v[4 * q + 0] = t.x;
            v[4 * q + 1] = t.y;
            v[4 * q + 2] = t.z;
            v[4 * q + 3] = t.w;
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] = (k0 + c < kend) ? A[sidx<UPPER>(i, k0 + c, lda)] : 0.f;
}

// Row `row` of the operand panel: the 32 values split into tf32 hi and lo parts, 16-byte chunks
// at their 128-byte-swizzle positions.
__device__ __forceinline__ void panel_row(unsigned char *hi, unsigned char *lo, int row, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 h4, l4;
        tc::split_tf32(x[4 * q + 0], h4.x, l4.x);
        tc::split_tf32(x[4 * q + 1], h4.y, l4.y);
        tc::split_tf32(x[4 * q + 2], h4.z, l4.z);
        tc::split_tf32(x[4 * q + 3], h4.w, l4.w);
        const uint32_t off = tc::sw128_offset(row, 4 * q);
        *reinterpret_cast<float4 *>(hi + off) = h4;
        *reinterpret_cast<float4 *>(lo + off) = l4;
    }
}

// One element of a panel row: its tf32 hi and lo parts at (row, k).
__device__ __forceinline__ void panel_elem(unsigned char *hi, unsigned char *lo, int row, int k, float x) {
    float h, l;
    tc::split_tf32(x, h, l);
    const uint32_t off = tc::sw128_offset(row, k);
    *reinterpret_cast<float *>(hi + off) = h;
    *reinterpret_cast<float *>(lo + off) = l;
}

// D[:, 0:N) (+)= A * B^T over K = 32 with the 3xTF32 split (hi*hi + hi*lo + lo*hi): A is 128 rows
// at a_hi / a_lo, B is N rows at b_hi / b_lo (shared-memory addresses of 128-byte-swizzled
// K-major tiles). `acc` false overwrites D on the first product.
__device__ __forceinline__ void mma_k32(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo, int N,
                                        bool acc) {
    const uint32_t idesc = tc::idesc_tf32(128, N);
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        tc::mma_tf32(d, tc::sdesc_sw128(a_hi + 32 * st), tc::sdesc_sw128(b_hi + 32 * st), idesc, acc || st > 0);
        tc::mma_tf32(d, tc::sdesc_sw128(a_hi + 32 * st), tc::sdesc_sw128(b_lo + 32 * st), idesc, true);
        tc::mma_tf32(d, tc::sdesc_sw128(a_lo + 32 * st), tc::sdesc_sw128(b_hi + 32 * st), idesc, true);
    }
}

// One step j of the diagonal-block factor (lane = row) in a shifting register frame: on entry
// a[m] is column j+m of this lane's row, updated by every column before j except column j-1's
// contribution to columns j+3 and beyond, which is applied here ("delayed") from column j-1 as
// published in shared memory (cvp[m] = L(j-1+m, j-1)) and this lane's lp = L(lane, j-1). The
// pivot chain never waits on shared memory: L(j+1, j) and L(j+2, j) come by shuffles, and the
// next pivot, A(j+1,j+1) - L(j+1,j)^2, is formed by its own lane and broadcast into d. The delayed
// FMAs depend only on the previous step, so they fill the chain's latency. On exit the frame has
// moved by one column. Column j of L goes to sLs[j*32 + m] = L(j+m, j), 1/L(j,j) to sRs[j].
template <bool FIRST>
__device__ __forceinline__ void factor_step(float (&a)[32], float &lp, int lane, int j, int kq, float &d,
                                            unsigned &failed, float *sLs, float *sRs) {
    float cvp[32];
    if (FIRST) {
#pragma unroll
        for (int m = 0; m < 32; ++m) cvp[m] = 0.f;
    } else {
        const float4 *c4 = reinterpret_cast<const float4 *>(sLs + (j - 1) * 32);
#pragma unroll
        for (int m4 = 0; m4 < 8; ++m4) {
            const float4 v4 = c4[m4];
            cvp[4 * m4 + 0] = v4.x;
            cvp[4 * m4 + 1] = v4.y;
            cvp[4 * m4 + 2] = v4.z;
            cvp[4 * m4 + 3] = v4.w;
        }
    }
    const bool ok = d > 0.f;
    const float rs = ok ? rsqrtf(d) : 0.f;
    failed |= (ok || j >= kq) ? 0u : (1u << j);
    const float l = (lane == j) ? (ok ? d * rs : d) : (lane > j ? a[0] * rs : 0.f);
    if (lane >= j) sLs[j * 32 + (lane - j)] = l;
    if (lane == 0) sRs[j] = rs;
    const float l1 = __shfl_sync(0xffffffffu, l, (j + 1) & 31);   // L(j+1, j); 0 past the block
    const float l2 = __shfl_sync(0xffffffffu, l, (j + 2) & 31);   // L(j+2, j)
    d = __shfl_sync(0xffffffffu, fmaf(-l, l, a[1]), (j + 1) & 31);   // lane j+1: its next pivot
    const float n0 = fmaf(-l, l1, a[1]);
    const float n1 = fmaf(-l, l2, fmaf(-lp, cvp[3], a[2]));
#pragma unroll
    for (int p = 2; p < 30; ++p) a[p] = fmaf(-lp, cvp[p + 2], a[p + 1]);   // column j+1+p, delayed
    a[30] = a[31];                                   // column j+31: valid only for j = 0 (lp = 0)
    a[31] = 0.f;
    a[0] = n0;
    a[1] = n1;
    lp = l;
    __syncwarp();                                    // column j is published for the next step
}

// One step of the inverse (column `lane` of Linv, shifting frame of F live rows): acc[0] is row
// k of the running right-hand side; Linv(k, lane) = acc[0] / L(k,k) goes, split, to row k of the
// operand tile; the later rows subtract L(k+m, k) * Linv(k, lane).
template <int F>
__device__ __forceinline__ void invert_step(float (&acc)[32], int lane, int k, const float *sLs, const float *sRs,
                                            unsigned char *b_hi, unsigned char *b_lo) {
    const float y = acc[0] * sRs[k];
    const float4 *c4 = reinterpret_cast<const float4 *>(sLs + k * 32);
#pragma unroll
    for (int m4 = 0; m4 < (F + 3) / 4; ++m4) {
        const float4 v4 = c4[m4];
        const float cv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = 4 * m4 + e;
            if (m == 0 || m >= F) continue;
            acc[m - 1] = fmaf(-y, cv[e], acc[m]);
        }
    }
    acc[F - 1] = 0.f;
    panel_elem(b_hi, b_lo, k, lane, y);
}

// Factor the 32 x 32 diagonal block held by one warp (lane = row; padding rows are identity),
// right-looking, one column per step (the step above) in a loop unrolled by four: a single warp
// issues in order, and four steps in one body let the compiler fill each step's pivot-chain
// latency with the neighbouring steps' independent FMAs and loads (micro-benchmark, one warp per
// SM: 248 -> 184 cycles per step; by two 265, by eight 180); inside the kernel, where the other
// warps share the issue slots, the whole factorisation moved by about 1% (f32 n=512 b1024). The
// body stays small enough for the instruction cache, which the fully unrolled factor was not.
// Returns the failure bit mask.
// Every 4 columns (and after the last) the column count `ready` becomes base + j + 1 (a
// block-scope release), so a second warp can invert the block a few columns behind.
__device__ __forceinline__ unsigned factor_diag(float (&a)[32], int lane, int kq, float *sLs, float *sRs, int *ready,
                                                int base) {
    unsigned failed = 0;
    float lp = 0.f;
    float d = __shfl_sync(0xffffffffu, a[0], 0);
    factor_step<true>(a, lp, lane, 0, kq, d, failed, sLs, sRs);
#pragma unroll 4
    for (int j = 1; j < 32; ++j) {
        factor_step<false>(a, lp, lane, j, kq, d, failed, sLs, sRs);
        if ((j & 3) == 3 && lane == 0) {
            __threadfence_block();
            *reinterpret_cast<volatile int *>(ready) = base + j + 1;
        }
    }
    return failed;
}

// Inverse of the factored diagonal block, Linv = L11^-1 (lower triangular), by one warp: lane c
// forward-substitutes the unit vector e_c with the columns of L11 from sLs / sRs (in a shifting
// frame like the factor's), producing column c of Linv; Linv(k, c) is stored split into tf32 hi and lo at row k, K
// index c of a 32-row operand tile, so the tile holds Linv row by row (the B operand of
// X = V * Linv^T). The frame narrows by 8 every 8 steps (32, 24, 16, 8 live rows), so no work is
// spent on rows already finished.
//
// Runs on a second warp while the factor is still in progress: before step k it waits (bounded)
// until the column count `ready` exceeds base + k. Returns false if a wait gave up.
__device__ __forceinline__ bool wait_column(const int *ready, int target, uint32_t max_polls) {
    for (uint32_t i = 0; i < max_polls; ++i) {
        if (*reinterpret_cast<const volatile int *>(ready) > target) {
            __threadfence_block();
            return true;
        }
        __nanosleep(32);                             // keep the polling off the shared-memory pipe
    }
    return false;
}

__device__ __forceinline__ bool invert_diag(int lane, const float *sLs, const float *sRs, unsigned char *b_hi,
                                            unsigned char *b_lo, const int *ready, int base) {
    constexpr uint32_t kPolls = 1u << 22;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = (i == lane) ? 1.f : 0.f;
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
        if (!wait_column(ready, base + k, kPolls)) return false;
        invert_step<32>(acc, lane, k, sLs, sRs, b_hi, b_lo);
    }
#pragma unroll 1
    for (int k = 8; k < 16; ++k) {
        if (!wait_column(ready, base + k, kPolls)) return false;
        invert_step<24>(acc, lane, k, sLs, sRs, b_hi, b_lo);
    }
#pragma unroll 1
    for (int k = 16; k < 24; ++k) {
        if (!wait_column(ready, base + k, kPolls)) return false;
        invert_step<16>(acc, lane, k, sLs, sRs, b_hi, b_lo);
    }
#pragma unroll 1
    for (int k = 24; k < 32; ++k) {
        if (!wait_column(ready, base + k, kPolls)) return false;
        invert_step<8>(acc, lane, k, sLs, sRs, b_hi, b_lo);
    }
    return true;
}

// S(i, k0 + c) = v[c] for c < cend (Upper with `vec` and a whole row: eight 16-byte stores).
template <bool UPPER>
__device__ __forceinline__ void store_row(float *A, int64_t lda, int i, int k0, int cend, const float (&v)[32],
                                          bool vec) {
    if (UPPER && vec && cend == 32) {
        float4 *p = reinterpret_cast<float4 *>(A + static_cast<int64_t>(i) * lda + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q) p[q] = make_float4(v[4 * q + 0], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        return;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c)
        if (c < cend) A[sidx<UPPER>(i, k0 + c, lda)] = v[c];
}

}  // namespace colblk

template <typename T, bool UPPER>
__global__ void __launch_bounds__(256, 1) colblock_kernel(const BatchArgs args) {
    static_assert(sizeof(T) == 4 && !is_cplx<T>::value, "column-block tensor-core kernel: f32");
    using C = ColBlkCfg;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *p_hi = sm + C::P0_HI;
    unsigned char *p_lo = sm + C::P0_LO;
    float *sLs = reinterpret_cast<float *>(sm + C::OFF_L11);
    float *sRs = reinterpret_cast<float *>(sm + C::OFF_RS);
    __shared__ uint32_t s_tmem;
    __shared__ uint64_t s_mbar[2];                 // MMA completion, per operand panel
    __shared__ int s_stop;     // 0 running, 2 a bounded wait gave up
    __shared__ int s_diag;     // failing column of the current diagonal block, -1 none
    __shared__ int s_ready;    // diagonal-block columns published so far (all slices)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t mat = blockIdx.x;
    const int n = args.n;
    float *A = static_cast<T *>(args.A) + mat * args.stride_a;
    const int64_t lda = args.lda;
    // 16-byte aligned rows of S (Upper): aligned base and item stride, lda a multiple of 4
    const bool vec = UPPER && (lda % 4 == 0) && (args.stride_a % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(args.A) & 15) == 0);
    if (args.mode != MODE_POTRF) return;      // factor-only variant (the dispatcher never asks otherwise)

    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&s_mbar[0], 1);
        tc::mbar_init(&s_mbar[1], 1);
        tc::mbar_fence_init();
        s_stop = 0;
        s_ready = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t s_base = tc::smem_u32(sm);
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;   // this warp's tensor-memory lanes
    constexpr uint32_t kPolls = 1u << 24;
    uint32_t phase = 0;                      // bit b: parity to wait for on panel b's mbarrier
    uint32_t pend = 0;                       // bit b: a committed batch reading panel b not yet waited for
    int lost = -1;                           // panel whose wait gave up here (its batch may still run)
    // wait for the last committed batch that reads panel b (every thread polls the mbarrier;
    // bounded). A wait that gives up flags the item; no further MMAs are issued after the next
    // barrier.
    auto wait_mma = [&](int b) {
        if (pend & (1u << b)) {
            if (tc::mbar_wait(&s_mbar[b], (phase >> b) & 1u, kPolls)) phase ^= 1u << b;
            else { s_stop = 2; lost = b; }
            pend &= ~(1u << b);
        }
        tc::fence_after_sync();
    };

    // rows of the block column owned by this thread (block-relative) and their row tiles; the
    // tile's tensor-memory lanes 32*(warp&3).. are the ones this warp may read
    const int rA = tid, rB = tid + 256;
    const int tA = warp >> 2, tB = 2 + (warp >> 2);
    bool stop = false;
    int slice_no = 0;

    for (int C0 = 0; C0 < n && !stop; C0 += C::W) {
        const int M = n - C0;
        const int Wb = M < C::W ? M : C::W;
        const int mtiles = (M + 127) >> 7;
        const int Nb = (Wb + 15) & ~15;      // MMA N: a multiple of 16 (columns past Wb are unused)

        // ---------------------------------------------- 1. block update from the finished columns
        const int nk = C0 >> 5;
        if (nk > 0) {
            // chunk kc is staged into panel kc&1 while the MMAs of chunk kc-1 run; each chunk's
            // rows are loaded two chunks ahead into one of two register buffers, so the global
            // load latency overlaps a whole chunk step
            auto step = [&](int kc, const float (&xa)[32], const float (&xb)[32]) {
                const int pb = kc & 1;
                wait_mma(pb);                                // chunk kc-2's MMAs are done: panel pb is free
                unsigned char *bh = sm + (pb ? C::P1_HI : C::P0_HI), *bl = sm + (pb ? C::P1_LO : C::P0_LO);
                if (rA < M) colblk::panel_row(bh, bl, rA, xa);
                if (rB < M) colblk::panel_row(bh, bl, rB, xb);
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncthreads();
                tc::fence_after_sync();
                if (s_stop) { stop = true; return; }         // uniform: read after the barrier
                if (tid == 0) {
                    const uint32_t ph = s_base + static_cast<uint32_t>(pb ? C::P1_HI : C::P0_HI);
                    const uint32_t pl = s_base + static_cast<uint32_t>(pb ? C::P1_LO : C::P0_LO);
                    for (int t = 0; t < mtiles; ++t)     // B: the block's own rows, the panel's first Nb
                        colblk::mma_k32(tmem + static_cast<uint32_t>(t * 128), ph + 16384u * t, pl + 16384u * t, ph, pl,
                                        Nb, kc > 0);
                    tc::mma_commit(&s_mbar[pb]);
                }
                pend |= 1u << pb;
            };
            auto fetch = [&](int kc, float (&xa)[32], float (&xb)[32]) {
                colblk::load_row<UPPER>(A, lda, C0 + rA, 32 * kc, rA < M ? 32 * (kc + 1) : 0, xa, vec);
                colblk::load_row<UPPER>(A, lda, C0 + rB, 32 * kc, rB < M ? 32 * (kc + 1) : 0, xb, vec);
            };
            float xa0[32], xb0[32], xa1[32], xb1[32];
            fetch(0, xa0, xb0);
            if (nk > 1) fetch(1, xa1, xb1);
            for (int kc = 0; kc < nk && !stop; kc += 2) {
                step(kc, xa0, xb0);
                if (stop) break;
                if (kc + 2 < nk) fetch(kc + 2, xa0, xb0);
                if (kc + 1 < nk) {
                    step(kc + 1, xa1, xb1);
                    if (stop) break;
                    if (kc + 3 < nk) fetch(kc + 3, xa1, xb1);
                }
            }
        }

        // ---------------------------------------------- 2. factor the block column, 32 columns at a time
        for (int q = 0; 32 * q < Wb && !stop; ++q) {
            const int Q0 = C0 + 32 * q;
            const int kq = min(32, n - Q0);
            const int rlo = 32 * q;                          // the slice's diagonal rows start here
            const bool liveA = rA >= rlo && rA < M, liveB = rB < M;
            float va[32], vb[32];
            colblk::load_row<UPPER>(A, lda, C0 + rA, Q0, liveA ? Q0 + kq : 0, va, vec);
            colblk::load_row<UPPER>(A, lda, C0 + rB, Q0, liveB ? Q0 + kq : 0, vb, vec);
            wait_mma(0);
            wait_mma(1);
            if (C0 > 0 || q > 0) {                           // the accumulator holds this slice's update
                if (tA < mtiles && (warp >= 4 || warp >= q)) {
                    float d[32];
                    tc::tmem_ld32(tmem + lane_base + static_cast<uint32_t>(tA * 128 + 32 * q), d);
#pragma unroll
                    for (int c = 0; c < 32; ++c) va[c] -= d[c];
                }
                if (tB < mtiles) {
                    float d[32];
                    tc::tmem_ld32(tmem + lane_base + static_cast<uint32_t>(tB * 128 + 32 * q), d);
#pragma unroll
                    for (int c = 0; c < 32; ++c) vb[c] -= d[c];
                }
            }
            if (kq < 32) {                                   // ragged last slice: no values past n
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (c >= kq) va[c] = 0.f;
                    if (c >= kq) vb[c] = 0.f;
                }
            }
            const bool solA = rA >= rlo + 32 && rA < M;     // rows below the diagonal block
            // diagonal block: warp q holds its rows (lane l = row Q0 + l; padding rows are identity),
            // factors and stores them; warp 4 + (q+1)%4 (on another scheduler) inverts L11 into the
            // B tile of the solve one column behind; the other rows go, split, into the panel (the
            // A operand of the solve)
            const int base = 32 * slice_no++;
            if (warp == q) {
                if (liveB) colblk::panel_row(p_hi, p_lo, rB, vb);   // this warp's lower rows first
                float a[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) a[c] = (lane < kq) ? (c <= lane ? va[c] : 0.f) : (c == lane ? 1.f : 0.f);
                const unsigned failed = colblk::factor_diag(a, lane, kq, sLs, sRs, &s_ready, base);
                if (lane == 0) s_diag = failed ? __ffs(failed) - 1 : -1;
            } else {
                if (solA) colblk::panel_row(p_hi, p_lo, rA, va);
                if (liveB) colblk::panel_row(p_hi, p_lo, rB, vb);
                if (warp == 4 + ((q + 1) & 3)) {
                    if (!colblk::invert_diag(lane, sLs, sRs, sm + C::OFF_BI_HI, sm + C::OFF_BI_LO, &s_ready, base))
                        s_stop = 2;
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            // the diagonal block's lower part, from its published columns (columns before a failure
            // are final), stored by warp q; after the solve's MMAs are issued when there is no failure
            auto store_diag = [&]() {
                if (warp == q && lane < kq) {
#pragma unroll 1
                    for (int c = 0; c <= lane; ++c) A[colblk::sidx<UPPER>(Q0 + lane, Q0 + c, lda)] = sLs[c * 32 + lane - c];
                }
            };
            if (s_stop || s_diag >= 0) {                     // uniform: read after the barrier
                store_diag();
                if (tid == 0 && !s_stop) args.info[mat] = Q0 + s_diag + 1;
                stop = true;
                break;
            }
            // L21 = A21 * L11^-T = V * Linv^T on the tensor cores, into this slice's accumulator
            // columns (their update was consumed above)
            if (tid == 0) {
                for (int t = 0; t < mtiles; ++t)
                    colblk::mma_k32(tmem + static_cast<uint32_t>(t * 128 + 32 * q), s_base + static_cast<uint32_t>(C::P0_HI) + 16384u * t,
                                    s_base + static_cast<uint32_t>(C::P0_LO) + 16384u * t,
                                    s_base + static_cast<uint32_t>(C::OFF_BI_HI), s_base + static_cast<uint32_t>(C::OFF_BI_LO),
                                    32, false);
                tc::mma_commit(&s_mbar[0]);
            }
            pend |= 1u;
            store_diag();
            wait_mma(0);
            const bool next = 32 * (q + 1) < Wb;             // the block has further slices
            const bool xA = tA < mtiles && (warp >= 4 || warp > q), xB = tB < mtiles;   // warp-uniform
            if (xA) tc::tmem_ld32(tmem + lane_base + static_cast<uint32_t>(tA * 128 + 32 * q), va);
            if (xB) tc::tmem_ld32(tmem + lane_base + static_cast<uint32_t>(tB * 128 + 32 * q), vb);
            if (next) {
                if (solA) colblk::panel_row(p_hi, p_lo, rA, va);
                if (liveB) colblk::panel_row(p_hi, p_lo, rB, vb);
            }
            if (next) {
                // D[:, 32(q+1) : Nb) += L21 * L21^T over this slice: A = every row tile of the
                // panel, B = the panel rows of the block's remaining columns
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncthreads();
                tc::fence_after_sync();
                if (tid == 0) {
                    const int c1 = 32 * (q + 1);
                    const uint32_t ph = s_base + static_cast<uint32_t>(C::P0_HI), pl = s_base + static_cast<uint32_t>(C::P0_LO);
                    for (int t = 0; t < mtiles; ++t)
                        colblk::mma_k32(tmem + static_cast<uint32_t>(t * 128 + c1), ph + 16384u * t, pl + 16384u * t,
                                        ph + 128u * c1, pl + 128u * c1, Nb - c1, C0 > 0 || q > 0);
                    tc::mma_commit(&s_mbar[0]);
                }
                pend |= 1u;
            } else {
                tc::fence_before_sync();
                __syncthreads();                             // L11 and the panel are free again
                tc::fence_after_sync();
            }
            // the solved rows go to global memory while the tensor cores run the update above
            if (solA) colblk::store_row<UPPER>(A, lda, C0 + rA, Q0, kq, va, vec);
            if (liveB) colblk::store_row<UPPER>(A, lda, C0 + rB, Q0, kq, vb, vec);
        }
    }
    wait_mma(0);
    wait_mma(1);
    // A thread whose wait gave up polls once more for that batch (no MMA was issued after it gave
    // up: the issuing thread reads s_stop after the next barrier). The outcome is published
    // through shared memory behind a barrier, so every thread takes the same path below; the item
    // reports -1 whenever any wait gave up, and the tensor memory is released either way.
    if (lost >= 0 && !tc::mbar_wait(&s_mbar[lost], (phase >> lost) & 1u, kPolls)) s_stop = 2;
    __syncthreads();
    if (tid == 0) {
        if (s_stop == 2) args.info[mat] = -1;
        else if (!stop) args.info[mat] = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace bl
