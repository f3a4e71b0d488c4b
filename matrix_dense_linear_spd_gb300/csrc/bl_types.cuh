// Scalar types and the few arithmetic helpers the kernels share.
//
// Complex values are interleaved (re, im) pairs, matching the C ABI's storage. Every helper is
// a plain restatement of complex arithmetic; the products that appear in Cholesky are
// a*conj(b) (the Hermitian rank-1 update) and a*b (back substitution in conjugated form).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace bl {

struct __align__(8) cf32 { float x, y; };
struct __align__(16) cf64 { double x, y; };

template <typename T> struct real_of { using type = T; };
template <> struct real_of<cf32> { using type = float; };
template <> struct real_of<cf64> { using type = double; };
template <typename T> using real_t = typename real_of<T>::type;

template <typename T> struct is_cplx { static constexpr bool value = false; };
template <> struct is_cplx<cf32> { static constexpr bool value = true; };
template <> struct is_cplx<cf64> { static constexpr bool value = true; };

__device__ __forceinline__ float re(float v) { return v; }
__device__ __forceinline__ double re(double v) { return v; }
__device__ __forceinline__ float re(cf32 v) { return v.x; }
__device__ __forceinline__ double re(cf64 v) { return v.x; }

__device__ __forceinline__ float im_part(float) { return 0.f; }
__device__ __forceinline__ double im_part(double) { return 0.0; }
__device__ __forceinline__ float im_part(cf32 v) { return v.y; }
__device__ __forceinline__ double im_part(cf64 v) { return v.y; }

template <typename T> __device__ __forceinline__ T zero();
template <> __device__ __forceinline__ float zero<float>() { return 0.f; }
template <> __device__ __forceinline__ double zero<double>() { return 0.0; }
template <> __device__ __forceinline__ cf32 zero<cf32>() { return {0.f, 0.f}; }
template <> __device__ __forceinline__ cf64 zero<cf64>() { return {0.0, 0.0}; }

template <typename T> __device__ __forceinline__ T from_real(real_t<T> r);
template <> __device__ __forceinline__ float from_real<float>(float r) { return r; }
template <> __device__ __forceinline__ double from_real<double>(double r) { return r; }
template <> __device__ __forceinline__ cf32 from_real<cf32>(float r) { return {r, 0.f}; }
template <> __device__ __forceinline__ cf64 from_real<cf64>(double r) { return {r, 0.0}; }

__device__ __forceinline__ float conj(float v) { return v; }
__device__ __forceinline__ double conj(double v) { return v; }
__device__ __forceinline__ cf32 conj(cf32 v) { return {v.x, -v.y}; }
__device__ __forceinline__ cf64 conj(cf64 v) { return {v.x, -v.y}; }

__device__ __forceinline__ float scale(float v, float r) { return v * r; }
__device__ __forceinline__ double scale(double v, double r) { return v * r; }
__device__ __forceinline__ cf32 scale(cf32 v, float r) { return {v.x * r, v.y * r}; }
__device__ __forceinline__ cf64 scale(cf64 v, double r) { return {v.x * r, v.y * r}; }

// acc -= a * conj(b)
__device__ __forceinline__ void sub_mul_conj(float &acc, float a, float b) { acc = fmaf(-a, b, acc); }
__device__ __forceinline__ void sub_mul_conj(double &acc, double a, double b) { acc = fma(-a, b, acc); }
__device__ __forceinline__ void sub_mul_conj(cf32 &acc, cf32 a, cf32 b) {
    acc.x = fmaf(-a.x, b.x, acc.x);
    acc.x = fmaf(-a.y, b.y, acc.x);
    acc.y = fmaf(-a.y, b.x, acc.y);
    acc.y = fmaf(a.x, b.y, acc.y);
}
__device__ __forceinline__ void sub_mul_conj(cf64 &acc, cf64 a, cf64 b) {
    acc.x = fma(-a.x, b.x, acc.x);
    acc.x = fma(-a.y, b.y, acc.x);
    acc.y = fma(-a.y, b.x, acc.y);
    acc.y = fma(a.x, b.y, acc.y);
}

// acc -= |a|^2 (acc real)
__device__ __forceinline__ void sub_abs2(float &acc, float a) { acc = fmaf(-a, a, acc); }
__device__ __forceinline__ void sub_abs2(double &acc, double a) { acc = fma(-a, a, acc); }
__device__ __forceinline__ void sub_abs2(float &acc, cf32 a) { acc = fmaf(-a.y, a.y, fmaf(-a.x, a.x, acc)); }
__device__ __forceinline__ void sub_abs2(double &acc, cf64 a) { acc = fma(-a.y, a.y, fma(-a.x, a.x, acc)); }

// acc -= a * b
__device__ __forceinline__ void sub_mul(float &acc, float a, float b) { acc = fmaf(-a, b, acc); }
__device__ __forceinline__ void sub_mul(double &acc, double a, double b) { acc = fma(-a, b, acc); }
__device__ __forceinline__ void sub_mul(cf32 &acc, cf32 a, cf32 b) {
    acc.x = fmaf(-a.x, b.x, acc.x);
    acc.x = fmaf(a.y, b.y, acc.x);
    acc.y = fmaf(-a.x, b.y, acc.y);
    acc.y = fmaf(-a.y, b.x, acc.y);
}
__device__ __forceinline__ void sub_mul(cf64 &acc, cf64 a, cf64 b) {
    acc.x = fma(-a.x, b.x, acc.x);
    acc.x = fma(a.y, b.y, acc.x);
    acc.y = fma(-a.x, b.y, acc.y);
    acc.y = fma(-a.y, b.x, acc.y);
}

// a += b
__device__ __forceinline__ void add_into(float &a, float b) { a += b; }
__device__ __forceinline__ void add_into(double &a, double b) { a += b; }
__device__ __forceinline__ void add_into(cf32 &a, cf32 b) { a.x += b.x; a.y += b.y; }
__device__ __forceinline__ void add_into(cf64 &a, cf64 b) { a.x += b.x; a.y += b.y; }

__device__ __forceinline__ float rsqrt_of(float d) { return rsqrtf(d); }
__device__ __forceinline__ double rsqrt_of(double d) { return rsqrt(d); }

// Asynchronous global -> shared copies (cp.async): no register round trip; completion by
// commit groups.
__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
template <int BYTES>
__device__ __forceinline__ void cp_async_elem(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(smem_addr(dst)), "l"(src), "n"(BYTES)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
// wait until at most N of this thread's most recent commit groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Operation selector shared by the kernels.
enum Mode : int { MODE_POTRF = 0, MODE_POSV = 1, MODE_POTRS = 2 };

// Launch parameters common to every family (sizes in elements of the dtype).
struct BatchArgs {
    int n;
    int nrhs;        // right-hand sides handled by this launch (0 for potrf)
    int mode;        // Mode
    int upper;       // 0 = Lower, 1 = Upper
    int64_t batch;
    void *A;
    int64_t lda, stride_a;
    void *B;
    int64_t ldb, stride_b;
    int32_t *info;   // may be null for MODE_POTRS
};

}  // namespace bl
