// Diagnostic: arithmetic peak microbenchmarks, so every roofline fraction of the library can be
// taken against a rate measured on the GPU it runs on rather than a datasheet figure.
//
// Each kernel keeps one execution unit busy with independent work and nothing else (no global
// memory traffic in the timed loop); the caller times the launch with CUDA events and divides the
// kernel's flop count by the time:
//   BL_PEAK_FFMA   FP32 fused multiply-add, scalar (fma.rn.f32): 2 flops per lane-instruction
//   BL_PEAK_FFMA2  FP32 packed pairs (fma.rn.f32x2): 4 flops per lane-instruction
//   BL_PEAK_DFMA   FP64 fused multiply-add: 2 flops per lane-instruction
//   BL_PEAK_DMMA   FP64 warp-level MMA (mma.sync m16n8k4 .f64): 1024 flops per warp-instruction
//   BL_PEAK_TF32   tcgen05.mma kind::tf32, M = 128, N = 256, K = 8, one issuing thread per SM:
//                  524,288 flops per instruction
//   BL_PEAK_BF16   tcgen05.mma kind::f16 with bf16 operands, M = 128, N = 256, K = 16: 1,048,576
//                  flops per instruction (a calibration point against a library bf16 GEMM)
// The tensor-core kernels multiply operand tiles of pseudo-random values held in shared memory
// into a tensor-memory accumulator; completion is awaited through an mbarrier with a time limit (the kernel
// reports a timeout in *status instead of waiting forever).
#include <cuda_runtime.h>

#include "../../include/bl.h"
#include "tc_sm100.cuh"

namespace bl {
namespace peak {

constexpr int CHAINS = 8;   // independent accumulators per thread

__global__ void __launch_bounds__(256) ffma_kernel(float *out, int iters, float a, float b) {
    float acc[CHAINS];
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) acc[c] = static_cast<float>(threadIdx.x + c);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
            for (int c = 0; c < CHAINS; ++c) acc[c] = fmaf(acc[c], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) s += acc[c];
    if (s == 1.2345f) out[threadIdx.x] = s;     // never true for the inputs used; keeps the work live
}

__global__ void __launch_bounds__(256) ffma2_kernel(float *out, int iters, float a, float b) {
    float2 acc[CHAINS];
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) acc[c] = make_float2(static_cast<float>(threadIdx.x + c), static_cast<float>(c));
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
            for (int c = 0; c < CHAINS; ++c) acc[c] = __ffma2_rn(acc[c], a2, b2);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) s += acc[c].x + acc[c].y;
    if (s == 1.2345f) out[threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) dfma_kernel(double *out, int iters, double a, double b) {
    double acc[CHAINS];
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) acc[c] = static_cast<double>(threadIdx.x + c);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
            for (int c = 0; c < CHAINS; ++c) acc[c] = fma(acc[c], a, b);
    }
    double s = 0.0;
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) s += acc[c];
    if (s == 1.2345) out[threadIdx.x] = s;
}

// D(16x8) += A(16x4) * B(4x8), f64; four independent accumulator sets per warp.
__global__ void __launch_bounds__(256) dmma_kernel(double *out, int iters, double a, double b) {
    double d[4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[s][i] = static_cast<double>(threadIdx.x + s + i);
    const double a0 = a, a1 = b, b0 = a - b;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int s = 0; s < 4; ++s)
                asm volatile(
                    "mma.sync.aligned.m16n8k4.row.col.f64.f64.f64.f64 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
                    "{%0,%1,%2,%3};\n"
                    : "+d"(d[s][0]), "+d"(d[s][1]), "+d"(d[s][2]), "+d"(d[s][3])
                    : "d"(a0), "d"(a1), "d"(b0));
    }
    double t = 0.0;
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) t += d[s][i];
    if (t == 1.2345) out[threadIdx.x] = t;
}

// Instruction descriptor, kind::f16 with bf16 A and B, f32 D, both K-major (same field layout as
// the kind::tf32 descriptor: D format in bits 4-5, A and B formats in bits 7-9 and 10-12, N/8 in
// bits 17-22, M/16 in bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, 1, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
    return t;
}

// Wait for the mbarrier phase with the given parity, at most limit_ns of wall time.
__device__ __forceinline__ bool mbar_wait_timed(uint64_t *mbar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (true) {
        if (tc::mbar_wait(mbar, parity, 64)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// One CTA per SM; thread 0 issues `iters` x 4 MMAs (M = 128, N = 256, 32 bytes of K each) into a
// 128 x 256 f32 tensor-memory accumulator from 128-byte-swizzled K-major tiles.
template <bool BF16>
__global__ void __launch_bounds__(128) tc_kernel(int iters, int32_t *status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
    // A: 128 rows x 128 bytes (16 KB); B: 256 rows x 128 bytes (32 KB), filled with values in
    // [1, 2) of pseudo-random mantissa (f32 words for tf32, bf16 pairs for bf16), so the rate is
    // the one of real data rather than of zero operands
    for (int i = threadIdx.x; i < (48 * 1024) / 4; i += blockDim.x) {
        uint32_t h = static_cast<uint32_t>(i) * 2654435761u + 0x9E3779B9u * (blockIdx.x + 1);
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        const uint32_t w = BF16 ? (((h & 0x007Fu) | 0x3F80u) | ((((h >> 16) & 0x007Fu) | 0x3F80u) << 16))
                                : ((h & 0x007FFFFFu) | 0x3F800000u);
        reinterpret_cast<uint32_t *>(base)[i] = w;
    }
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_ok;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, 256);
        tc::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(&mbar, 1);
        tc::mbar_fence_init();
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0) {
        const uint32_t sa = tc::smem_u32(base), sb = sa + 16384;
        const uint32_t idesc = BF16 ? idesc_bf16(128, 256) : tc::idesc_tf32(128, 256);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                const uint64_t ad = tc::sdesc_sw128(sa + 32 * st), bd = tc::sdesc_sw128(sb + 32 * st);
                if (BF16) mma_bf16(tmem, ad, bd, idesc);
                else tc::mma_tf32(tmem, ad, bd, idesc, true);
            }
        }
        tc::mma_commit(&mbar);
        s_ok = mbar_wait_timed(&mbar, 0, 4000000000ull) ? 1 : 0;   // 4 s
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
    if (threadIdx.x == 0 && !s_ok) atomicExch(status, 2);
}

}  // namespace peak
}  // namespace bl

extern "C" bl_status bl_debug_peak(int kind, int blocks, int iters, void *scratch, int32_t *status,
                                   double *flops, bl_stream_t stream) {
    using namespace bl::peak;
    if (blocks < 1 || iters < 1 || !scratch || !status || !flops) return BL_ERR_INVALID_ARGUMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const double nb = static_cast<double>(blocks), ni = static_cast<double>(iters);
    switch (kind) {
    case BL_PEAK_FFMA:
        ffma_kernel<<<blocks, 256, 0, st>>>(static_cast<float *>(scratch), iters, 0.999f, 1e-3f);
        *flops = nb * 256 * ni * 16 * CHAINS * 2;
        break;
    case BL_PEAK_FFMA2:
        ffma2_kernel<<<blocks, 256, 0, st>>>(static_cast<float *>(scratch), iters, 0.999f, 1e-3f);
        *flops = nb * 256 * ni * 16 * CHAINS * 4;
        break;
    case BL_PEAK_DFMA:
        dfma_kernel<<<blocks, 256, 0, st>>>(static_cast<double *>(scratch), iters, 0.999, 1e-3);
        *flops = nb * 256 * ni * 16 * CHAINS * 2;
        break;
    case BL_PEAK_DMMA:
        dmma_kernel<<<blocks, 256, 0, st>>>(static_cast<double *>(scratch), iters, 0.999, 1e-3);
        *flops = nb * 8 * ni * 8 * 4 * (2.0 * 16 * 8 * 4);
        break;
    case BL_PEAK_TF32:
    case BL_PEAK_BF16: {
        const size_t smem = 48 * 1024 + 1024;
        const bool bf = kind == BL_PEAK_BF16;
        auto kern = bf ? tc_kernel<true> : tc_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return BL_ERR_CUDA;
        kern<<<blocks, 128, smem, st>>>(iters, status);
        *flops = nb * ni * 4 * (2.0 * 128 * 256 * (bf ? 16 : 8));
        break;
    }
    default:
        return BL_ERR_INVALID_ARGUMENT;
    }
    return cudaGetLastError() == cudaSuccess ? BL_SUCCESS : BL_ERR_CUDA;
}
