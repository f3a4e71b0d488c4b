// Diagnostic: one 128 x 128 output tile C = A * B^T (A, B: 128 x 32, f32, row-major) on the
// tensor cores with the 3xTF32 split (hi*hi + hi*lo + lo*hi), through exactly the descriptors,
// tensor-memory handling and completion protocol the column-block Cholesky's updates use.
// It exists so that layer can be checked in isolation against a host product.
#include <cuda_runtime.h>

#include "../../include/bl.h"
#include "tc_sm100.cuh"

namespace bl {

__global__ void __launch_bounds__(128) tc_tile_check_kernel(const float *A, const float *B, float *C,
                                                             int32_t *status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned operand tiles: A_hi, A_lo, B_hi, B_lo (16 KB each)
    unsigned char *base = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *a_hi = base, *a_lo = base + 16384, *b_hi = base + 32768, *b_lo = base + 49152;
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, 128);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&mbar, 1);
        tc::mbar_fence_init();
    }
    for (int idx = tid; idx < 128 * 32; idx += 128) {
        const int row = idx >> 5, k = idx & 31;
        float h, l;
        tc::split_tf32(A[idx], h, l);
        *reinterpret_cast<float *>(a_hi + tc::sw128_offset(row, k)) = h;
        *reinterpret_cast<float *>(a_lo + tc::sw128_offset(row, k)) = l;
        tc::split_tf32(B[idx], h, l);
        *reinterpret_cast<float *>(b_hi + tc::sw128_offset(row, k)) = h;
        *reinterpret_cast<float *>(b_lo + tc::sw128_offset(row, k)) = l;
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (tid == 0) {
        constexpr uint32_t idesc = tc::idesc_tf32(128, 128);
        const uint32_t sa_hi = tc::smem_u32(a_hi), sa_lo = tc::smem_u32(a_lo);
        const uint32_t sb_hi = tc::smem_u32(b_hi), sb_lo = tc::smem_u32(b_lo);
        for (int s = 0; s < 4; ++s)   // K = 32 in steps of 8 (32 bytes)
            tc::mma_tf32(tmem, tc::sdesc_sw128(sa_hi + 32 * s), tc::sdesc_sw128(sb_hi + 32 * s), idesc, s > 0);
        for (int s = 0; s < 4; ++s)
            tc::mma_tf32(tmem, tc::sdesc_sw128(sa_hi + 32 * s), tc::sdesc_sw128(sb_lo + 32 * s), idesc, true);
        for (int s = 0; s < 4; ++s)
            tc::mma_tf32(tmem, tc::sdesc_sw128(sa_lo + 32 * s), tc::sdesc_sw128(sb_hi + 32 * s), idesc, true);
        tc::mma_commit(&mbar);
    }
    const bool ok = tc::mbar_wait(&mbar, 0, 1u << 22);
    tc::fence_after_sync();
    if (!ok) {
        if (lane == 0) atomicExch(status, 2);   // the MMA never completed: report, do not hang
    } else {
        const int row = warp * 32 + lane;
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) C[row * 128 + c0 + i] = v[i];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    if (tid == 0 && ok) atomicCAS(status, 0, 1);
}

}  // namespace bl

extern "C" bl_status bl_debug_tc_tile_f32(const float *A, const float *B, float *C, int32_t *status,
                                          bl_stream_t stream) {
    if (!A || !B || !C || !status) return BL_ERR_INVALID_ARGUMENT;
    const size_t smem = 4 * 16384 + 1024;
    cudaError_t e = cudaFuncSetAttribute(bl::tc_tile_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return BL_ERR_CUDA;
    bl::tc_tile_check_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(A, B, C, status);
    return cudaGetLastError() == cudaSuccess ? BL_SUCCESS : BL_ERR_CUDA;
}
