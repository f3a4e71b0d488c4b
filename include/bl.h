/*
 * bl.h -- batched Cholesky factorisation and positive-definite solve for GB300 (sm_103a).
 *
 * C ABI of libbl.so. All matrices are column-major: element (i, j) of item b of a batch lives
 * at  base + b*stride + j*ld + i  (in elements of the dtype; complex elements are interleaved
 * real/imaginary pairs). Every pointer argument except `stream` is a DEVICE pointer owned by
 * the caller; the library allocates nothing, keeps no reference after the call returns, and
 * never synchronises the host: work is enqueued on `stream` (NULL = the legacy default stream)
 * and completes in stream order.
 *
 * Semantics follow the BatchLAS documentation pages:
 *   - "Batched Cholesky (potrf)", section "Selection" / "can_run() terms": A = L*L^H (Lower)
 *     or A = U^H*U (Upper) for each Hermitian positive-definite item; Upper is the same
 *     recurrence on S(i,c) = conj(A(c,i)), a load and store transform.
 *   - same page, "potrf: correctness findings" item 6: info[b] = 0 on success, otherwise the
 *     1-based index of the first pivot that is not positive (a NaN pivot fails too); a
 *     failure inside a panel is reported at its global column.
 *   - same page, "posv selection" and "The fused potrs solve": posv factors A and solves
 *     A*X = B with both triangular solves; B is overwritten by X.
 *
 * Numerical failure is not an error: the call returns BL_SUCCESS and reports it in info.
 * Argument errors are detected on the host before anything is enqueued and return
 * BL_ERR_INVALID_ARGUMENT with no side effects.
 */
#ifndef BL_H
#define BL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st*). NULL selects the legacy default stream. */
typedef struct CUstream_st *bl_stream_t;

typedef enum { BL_LOWER = 0, BL_UPPER = 1 } bl_uplo;

/* f32 = float, f64 = double, c64 = complex<float>, c128 = complex<double>. */
typedef enum { BL_F32 = 0, BL_F64 = 1, BL_C64 = 2, BL_C128 = 3 } bl_dtype;

typedef enum {
    BL_SUCCESS = 0,
    BL_ERR_INVALID_ARGUMENT = 1, /* bad size, stride, pointer, enum, or an unrunnable route pin */
    BL_ERR_NO_ROUTE = 2,         /* no kernel family can run the shape (only reachable by pins) */
    BL_ERR_CUDA = 3,             /* a CUDA launch or attribute call failed; see bl_last_error() */
    BL_ERR_INTERNAL = 4
} bl_status;

/*
 * bl_potrf -- factor `batch` independent n x n Hermitian positive-definite matrices in place.
 *
 *   uplo      BL_LOWER: read and overwrite the lower triangle (incl. diagonal) with L.
 *             BL_UPPER: read and overwrite the upper triangle with U. The other triangle is
 *             neither read for any result nor written.
 *   dtype     element type of A.
 *   n         order, n >= 1.           batch   number of items, batch >= 1.
 *   A         device pointer to item 0. lda >= n. stride_a >= lda*n (items do not overlap).
 *   info      device int32[batch]; receives 0 or the 1-based first failing column.
 *   stream    CUDA stream.
 *
 * A must be aligned to its element size (4, 8, 8 or 16 bytes for f32, f64, c64, c128) and info
 * to 4 bytes; lda and stride_a may take any value (16-byte aligned columns take faster copy
 * paths). For a failed item only info and the leading (info-1) x (info-1) block of the factor
 * are defined; the rest of the referenced triangle holds unspecified finite or non-finite
 * values. info[b] = -1 reports that the kernel gave up waiting for an asynchronous copy or
 * tensor-core operation of that item (a device fault, not a numerical result): the item's
 * outputs are undefined.
 */
bl_status bl_potrf(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t batch, void *A,
                   int64_t lda, int64_t stride_a, int32_t *info, bl_stream_t stream);

/*
 * bl_posv -- factor A as bl_potrf does, then solve A*X = B for nrhs right-hand sides per item
 * (forward substitution with L, back substitution with L^H; Upper uses U^H and U).
 *
 *   B         device pointer, n x nrhs per item, aligned to the element size, ldb >= n,
 *             stride_b >= ldb*nrhs. Overwritten
 *             by X for items whose factorisation succeeded; left untouched for failed items.
 *   nrhs      nrhs >= 1. Any nrhs is accepted; the fused kernels take up to 8 (or fewer,
 *             depending on the kernel) per pass and larger counts run in further passes of the
 *             solve-only kernel on the stored factor.
 * Other arguments as bl_potrf. A and B must not overlap.
 */
bl_status bl_posv(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t nrhs, int64_t batch,
                  void *A, int64_t lda, int64_t stride_a, void *B, int64_t ldb,
                  int64_t stride_b, int32_t *info, bl_stream_t stream);

/*
 * bl_potrs -- solve A*X = B given the Cholesky factor already stored in the `uplo` triangle of
 * A (as produced by bl_potrf). A is read only; B is overwritten by X. No info is produced: a
 * factor with a zero or non-finite diagonal gives non-finite X. Arguments as bl_posv.
 * (Source: "Batched Cholesky (potrf)", "The fused potrs solve": the solve-only kernel that posv
 * runs after the factorisation.)
 */
bl_status bl_potrs(bl_uplo uplo, bl_dtype dtype, int64_t n, int64_t nrhs, int64_t batch,
                   const void *A, int64_t lda, int64_t stride_a, void *B, int64_t ldb,
                   int64_t stride_b, bl_stream_t stream);

/* Static, human-readable name of a status code. */
const char *bl_status_string(bl_status status);

/* The calling thread's last error message (empty string if none). Valid until the next call
 * into the library from the same thread. */
const char *bl_last_error(void);

/* The calling thread's last routing decision, spelled "family[:field=value]..." (for example
 * "tile:p=4:s=8"), or "" before the first call. */
const char *bl_last_choice(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
int bl_version(void);

/*
 * Kernel selection controls (BatchLAS "Flat kernel selection", section 5.2: pins).
 *
 * bl_set_route pins the kernel variant for op "potrf", "posv" or "potrs" on the calling thread,
 * overriding the environment variables BL_POTRF_ROUTE / BL_POSV_ROUTE / BL_POTRS_ROUTE (read
 * once per process). `spelling` is a variant name as returned by bl_route_name, "auto" (table
 * selection), or NULL / "" to clear. A pin that names no variant, or one that cannot run the
 * shape of a later call, makes that call return BL_ERR_INVALID_ARGUMENT.
 */
bl_status bl_set_route(const char *op, const char *spelling);

/* Number of compiled kernel variants for `dtype`, and the spelling of variant i (NULL when i is
 * out of range; the string is valid until the next call on this thread). */
int bl_num_routes(bl_dtype dtype);
const char *bl_route_name(bl_dtype dtype, int i);

/* Capacity of variant i: returns the largest order it holds (for "tile" variants: n plus the
 * right-hand sides of one pass; for "warp" and "thread" variants: n; "thread:n=N:e=1" runs its
 * unrolled path at n = N and the general one below), 0 for "any order", or -1 when i is out of
 * range; *rhs_per_pass receives the right-hand sides one pass solves (0 = any, -1 = the variant
 * factors only: potrf, not posv or potrs). */
int bl_route_capacity(bl_dtype dtype, int i, int *rhs_per_pass);

/*
 * Selection without a GPU, for host-side tests of the selection layer: the choice that an op
 * (0 = potrf, 1 = posv, 2 = potrs) would make on a synthetic device with table key `devkey`
 * (for example "sm_103") and `smem_optin` bytes of opt-in shared memory per block. Makes no
 * CUDA call. Returns "<spelling> [<reason>]" or "error: <message>"; the string is valid until
 * the next call on this thread.
 */
const char *bl_select_debug(int op, bl_dtype dtype, bl_uplo uplo, int64_t n, int64_t nrhs,
                            int64_t batch, const char *devkey, int64_t smem_optin);

/*
 * Diagnostic: one 128 x 128 tile C = A * B^T on the tensor cores (tcgen05, kind::tf32) with the
 * 3xTF32 split the column-block factorisation's updates use. A and B are device pointers to
 * 128 x 32 row-major f32 matrices, C to a 128 x 128 row-major f32 result; *status (device int32,
 * initially 0) becomes 1 on completion or 2 if the tensor-core work did not complete within the
 * kernel's bounded wait. Launches one CTA on `stream`.
 */
bl_status bl_debug_tc_tile_f32(const float *A, const float *B, float *C, int32_t *status,
                               bl_stream_t stream);

/*
 * Diagnostic: arithmetic-peak microbenchmarks, so that roofline fractions can be taken against
 * rates measured on the device in use (the pages state their rooflines against measured
 * bandwidths and rates of the card under test: "Small-n baseline", the DRAM-roof paragraph).
 * Launches `blocks` CTAs of one kernel that keeps one execution unit busy for `iters` loop trips
 * and stores the kernel's total flop count in *flops (host pointer); the caller times the launch
 * (CUDA events on `stream`) and divides. `scratch` is a device buffer of at least 2 KB that the
 * kernels never write in practice (it keeps the arithmetic from being optimised away); *status
 * (device int32, initially 0) becomes 2 if a tensor-core kernel's bounded wait for its MMAs gave
 * up. Kinds:
 *   BL_PEAK_FFMA   FP32 fma.rn.f32, 256-thread CTAs         BL_PEAK_FFMA2  FP32 fma.rn.f32x2 pairs
 *   BL_PEAK_DFMA   FP64 fma                                 BL_PEAK_DMMA   FP64 mma.sync m16n8k4
 *   BL_PEAK_TF32   tcgen05.mma kind::tf32, 128x256x8, one CTA per SM (blocks = SM count)
 *   BL_PEAK_BF16   tcgen05.mma kind::f16 (bf16), 128x256x16, one CTA per SM
 */
typedef enum {
    BL_PEAK_FFMA = 0, BL_PEAK_FFMA2 = 1, BL_PEAK_DFMA = 2, BL_PEAK_DMMA = 3, BL_PEAK_TF32 = 4, BL_PEAK_BF16 = 5
} bl_peak_kind;
bl_status bl_debug_peak(int kind, int blocks, int iters, void *scratch, int32_t *status, double *flops,
                        bl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BL_H */
