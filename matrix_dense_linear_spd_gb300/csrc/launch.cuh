// Launch helpers and the registry entry type shared by the per-dtype instantiation files.
#pragma once

#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <cuda_runtime.h>

#include "bl_types.cuh"
#include "registry.h"
#include "blocked_kernel.cuh"
#include "colblock_kernel.cuh"
#include "tile_kernel.cuh"
#include "warp_kernel.cuh"
#include "warp2_kernel.cuh"
#include "thread_kernel.cuh"

namespace bl {

// Raise the dynamic shared-memory limit once per device for kernels above 48 KB.
template <typename K>
inline cudaError_t ensure_smem(K kern, size_t bytes, std::atomic<unsigned long long> &done) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <typename T, int P, int S>
cudaError_t launch_tile(const BatchArgs &a, cudaStream_t st) {
    using C = TileCfg<T, P, S>;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = ensure_smem(tile_kernel<T, P, S>, C::smem_bytes, done);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((a.batch + C::G - 1) / C::G);
    tile_kernel<T, P, S><<<grid, C::THREADS, C::smem_bytes, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int NB>
cudaError_t launch_blocked(const BatchArgs &a, cudaStream_t st) {
    using C = BlkCfg<T, NB>;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = ensure_smem(blocked_kernel<T, NB>, C::smem_bytes, done);
    if (e != cudaSuccess) return e;
    blocked_kernel<T, NB><<<static_cast<unsigned>(a.batch), C::THREADS, C::smem_bytes, st>>>(a);
    return cudaGetLastError();
}

// Persistent grid for the warp family: enough CTAs to fill every SM at the kernel's occupancy,
// never more than the work needs. The resident-CTA count is cached per kernel, device and
// shared-memory size (the occupancy query costs more than the launch itself).
template <typename K>
inline unsigned persistent_grid(K kern, int threads, size_t smem, int64_t ctas_needed) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, size_t>, long long> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const auto key = std::make_tuple(reinterpret_cast<const void *>(kern), dev, smem);
    long long full = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) full = it->second;
    }
    if (full <= 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
            per_sm = 1, sms = sms > 0 ? sms : 1;
        full = static_cast<long long>(sms) * per_sm;
        std::lock_guard<std::mutex> lk(mu);
        cache[key] = full;
    }
    return static_cast<unsigned>(ctas_needed < full ? ctas_needed : full);
}

// WHOLE: the "full=1" variant, which copies whole squares into its slabs when the call's items are
// stored back to back (n = N, lda = N, stride = N*N, 16-byte aligned) and otherwise runs the
// compacted-triangle kernel like the plain variant (same arithmetic, bit-identical results).
// PK: packed two-lane FP32 FMAs in the rank-1 update (f32), in both the factor-only and the
// solve kernels.
template <typename T, int P, int R, bool WHOLE = false, bool PK = false, bool LA = false, bool V2 = false>
cudaError_t launch_warp(const BatchArgs &a, cudaStream_t st) {
    using C = WarpCfg<T, P, R>;
    const int64_t groups = (a.batch + C::G - 1) / C::G;
    const int64_t ctas = (groups + C::WARPS - 1) / C::WARPS;
    // items stored back to back (n = N, lda = N, stride = N*N, 16-byte aligned): each group is one
    // contiguous run, copied whole into full-square slabs
    const bool full = WHOLE && a.n == C::N && a.lda == C::N &&
                      a.stride_a == static_cast<int64_t>(C::N) * C::N && (reinterpret_cast<uintptr_t>(a.A) & 15) == 0;
    if (a.mode == MODE_POTRF) {
        if constexpr (WHOLE && C::full_ok) {
            if constexpr (V2) {
                if (full) {   // float2-pair rows (f32); Upper stages its store
                    constexpr bool cs = C::v2_compact;
                    auto kern = warp2_kernel<P, R, cs ? C::min_blocks_v2c() : C::min_blocks_packed(), LA, false, cs>;
                    constexpr size_t sm_up = cs ? C::smem_potrf : C::smem_potrf_full;
                    const size_t sm = a.upper ? sm_up : (cs ? C::smem_lower : C::smem_full);
                    static std::atomic<unsigned long long> done{0};
                    cudaError_t e = ensure_smem(kern, sm_up, done);
                    if (e != cudaSuccess) return e;
                    kern<<<persistent_grid(kern, C::THREADS, sm, ctas), C::THREADS, sm, st>>>(a);
                    return cudaGetLastError();
                }
            }
            if (full) {
                auto kern = warp_kernel<T, P, R, false, PK ? C::min_blocks_packed() : C::min_blocks_full(), true, PK>;
                const size_t sm = a.upper ? C::smem_potrf_full : C::smem_full;   // Upper stages its store
                static std::atomic<unsigned long long> done{0};
                cudaError_t e = ensure_smem(kern, C::smem_potrf_full, done);
                if (e != cudaSuccess) return e;
                kern<<<persistent_grid(kern, C::THREADS, sm, ctas), C::THREADS, sm, st>>>(a);
                return cudaGetLastError();
            }
        }
        auto kern = warp_kernel<T, P, R, false, PK ? C::min_blocks_packed() : C::min_blocks(), false, PK>;
        const size_t sm = a.upper ? C::smem_potrf : C::smem_lower;  // Lower needs no staging slab
        static std::atomic<unsigned long long> done{0};
        cudaError_t e = ensure_smem(kern, C::smem_potrf, done);
        if (e != cudaSuccess) return e;
        kern<<<persistent_grid(kern, C::THREADS, sm, ctas), C::THREADS, sm, st>>>(a);
    } else {
        if constexpr (WHOLE && C::full_solve_ok && C::smem_solve_full <= 227 * 1024) {
            if constexpr (V2) {
                if (full && a.mode == MODE_POSV) {   // float2-pair rows, fused solve (first pass)
                    constexpr bool cs = C::v2_compact;
                    constexpr size_t sm = cs ? C::smem_solve : C::smem_solve_full;
                    auto kern = warp2_kernel<P, R, C::min_blocks_solve(sm), LA, true, cs>;
                    static std::atomic<unsigned long long> done{0};
                    cudaError_t e = ensure_smem(kern, sm, done);
                    if (e != cudaSuccess) return e;
                    kern<<<persistent_grid(kern, C::THREADS, sm, ctas), C::THREADS, sm, st>>>(a);
                    return cudaGetLastError();
                }
            }
            if (full) {
                auto kern = warp_kernel<T, P, R, true, C::min_blocks_solve(C::smem_solve_full), true, PK>;
                static std::atomic<unsigned long long> done{0};
                cudaError_t e = ensure_smem(kern, C::smem_solve_full, done);
                if (e != cudaSuccess) return e;
                kern<<<persistent_grid(kern, C::THREADS, C::smem_solve_full, ctas), C::THREADS, C::smem_solve_full, st>>>(a);
                return cudaGetLastError();
            }
        }
        auto kern = warp_kernel<T, P, R, true, C::min_blocks_solve(C::smem_solve), false, PK>;
        static std::atomic<unsigned long long> done{0};
        cudaError_t e = ensure_smem(kern, C::smem_solve, done);
        if (e != cudaSuccess) return e;
        kern<<<persistent_grid(kern, C::THREADS, C::smem_solve, ctas), C::THREADS, C::smem_solve, st>>>(a);
    }
    return cudaGetLastError();
}

// V2: the whole-square kernel with float2 column-pair rows (warp2_kernel.cuh) for potrf and the
// first pass of posv, LA with look-ahead pivots; other calls of such a variant (other layouts,
// solve-only passes) run the kernels of warp_kernel.cuh.
template <typename T, int P, int R, bool WHOLE = false, bool PK = false, bool LA = false, bool V2 = false>
constexpr KernelEntry warp_entry() {
    using C = WarpCfg<T, P, R>;
    static_assert(!WHOLE || C::full_ok, "whole-square slabs need whole 16-byte chunks per lane");
    static_assert(!V2 || (WHOLE && PK), "float2-pair rows: whole squares, packed update");
    static_assert(!LA || V2, "look-ahead pivots: float2-pair rows");
    return KernelEntry{2, P, R, (WHOLE ? 1 : 0) | (PK ? 2 : 0) | (LA ? 4 : 0) | (V2 ? 8 : 0), C::N, C::RHS, C::THREADS,
                       C::PER_CTA, WHOLE ? C::smem_solve_full : C::smem_solve, &launch_warp<T, P, R, WHOLE, PK, LA, V2>};
}

template <typename T, int NMAX, int TPMX, bool EXACT>
cudaError_t launch_thread(const BatchArgs &a, cudaStream_t st) {
    using C = ThreadCfg<T, NMAX, TPMX>;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = ensure_smem(thread_kernel<T, NMAX, TPMX, EXACT>, C::smem_bytes, done);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((a.batch + C::MATS - 1) / C::MATS);
    thread_kernel<T, NMAX, TPMX, EXACT><<<grid, C::THREADS, C::smem_bytes, st>>>(a);
    return cudaGetLastError();
}

// TPMX = 2: a pair of lanes per matrix ("thread:n=NMAX:p=2"); EXACT: fully unrolled at n == NMAX
// ("thread:n=NMAX:e=1")
template <typename T, int NMAX, int TPMX = 1, bool EXACT = false>
constexpr KernelEntry thread_entry() {
    static_assert(!EXACT || TPMX == 1, "the unrolled order-N factor is one lane per matrix");
    using C = ThreadCfg<T, NMAX, TPMX>;
    return KernelEntry{3, TPMX == 1 ? 0 : TPMX, EXACT ? 1 : 0, NMAX, NMAX, -1, C::THREADS, C::MATS, C::smem_bytes,
                       &launch_thread<T, NMAX, TPMX, EXACT>};
}

template <typename T, int P, int S>
constexpr KernelEntry tile_entry() {
    using C = TileCfg<T, P, S>;
    return KernelEntry{0, P, S, 0, C::N, P, C::THREADS, C::G, C::smem_bytes, &launch_tile<T, P, S>};
}

template <typename T>
cudaError_t launch_colblock(const BatchArgs &a, cudaStream_t st) {
    static std::atomic<unsigned long long> done{0};
    static std::atomic<unsigned long long> done_u{0};
    cudaError_t e = a.upper ? ensure_smem(colblock_kernel<T, true>, ColBlkCfg::smem_bytes, done_u)
                            : ensure_smem(colblock_kernel<T, false>, ColBlkCfg::smem_bytes, done);
    if (e != cudaSuccess) return e;
    if (a.upper)
        colblock_kernel<T, true><<<static_cast<unsigned>(a.batch), ColBlkCfg::THREADS, ColBlkCfg::smem_bytes, st>>>(a);
    else
        colblock_kernel<T, false><<<static_cast<unsigned>(a.batch), ColBlkCfg::THREADS, ColBlkCfg::smem_bytes, st>>>(a);
    return cudaGetLastError();
}

// The column-block tensor-core kernel (f32 potrf, n <= 512): blocked family, panel width 32,
// spelled with tc=2; factor only.
template <typename T>
constexpr KernelEntry colblock_entry() {
    return KernelEntry{1, 0, 2, 32, ColBlkCfg::MAXN, -1, ColBlkCfg::THREADS, 1, ColBlkCfg::smem_bytes,
                       &launch_colblock<T>};
}

template <typename T, int NB>
constexpr KernelEntry blocked_entry() {
    using C = BlkCfg<T, NB>;
    return KernelEntry{1, 0, 0, NB, 0, 0, C::THREADS, 1, C::smem_bytes, &launch_blocked<T, NB>};
}

}  // namespace bl
