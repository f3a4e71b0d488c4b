/*
 * CPU oracle for batched Cholesky (potrf) and the positive-definite solve (posv / potrs).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent reference that the CUDA library is
 * checked against. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the library itself never calls it and shares no code, header or constant with
 * it.
 *
 * It is a plain, unblocked, deliberately slow restatement of the textbook definitions, in
 * `long double` (80-bit x87 extended on x86-64, IEEE binary128 in software on aarch64):
 *
 *   potrf, Lower  -- Cholesky-Banachiewicz, row by row (source: BatchLAS "Batched Cholesky
 *                    (potrf)" page; the factor satisfies A = L*L^H, and the per-matrix info is
 *                    the 1-based index of the first pivot that is not positive, sections
 *                    "potrf: correctness findings" items 5-6 and "The pivot-cell WAR race").
 *                    For row i:  L(i,j) = (A(i,j) - sum_{k<j} L(i,k)*conj(L(j,k))) / L(j,j),
 *                    j < i;  d = Re A(i,i) - sum_{k<i} |L(i,k)|^2;  if !(d > 0) stop with
 *                    info = i+1 (NaN fails too), else L(i,i) = sqrt(d).
 *   potrf, Upper  -- the same recurrence on S(i,c) = conj(A(c,i)) read from the upper
 *                    triangle; the result is stored as U(c,i) = conj(L(i,c)), so A = U^H*U
 *                    (same page, "can_run() terms": Upper is a load and store transform).
 *   posv          -- after a successful factorisation, forward substitution L*y = b and back
 *                    substitution L^H*x = y for every right-hand side (same page, "The fused
 *                    potrs solve"). On failure the right-hand sides are returned unchanged.
 *   potrs         -- the two substitutions alone, given a factor.
 *
 * Inputs arrive as double / interleaved-complex double values (every f32, f64, c64 and c128
 * value promotes to double exactly) in the caller's column-major layout: element (i,j) of
 * item b at  b*stride + j*ld + i  (complex: twice that, in doubles). Outputs are long double.
 * The imaginary part of a complex diagonal entry of A is ignored, and the diagonal of the
 * factor is real (LAPACK convention).
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef long double ldr;
typedef long double complex ldc;

/* ---------------------------------------------------------------- element access helpers */

/* Read the referenced-triangle entry of the Hermitian input as the Lower recurrence sees it:
 * Lower reads A(i,c) for c <= i; Upper reads S(i,c) = conj(A(c,i)). */
static ldr in_real(const double *a, int64_t ld, int upper, int64_t i, int64_t c) {
    return upper ? (ldr)a[i * ld + c] : (ldr)a[c * ld + i];
}

static ldc in_cplx(const double *a, int64_t ld, int upper, int64_t i, int64_t c) {
    int64_t off = upper ? (i * ld + c) : (c * ld + i);
    ldr re = (ldr)a[2 * off], im = (ldr)a[2 * off + 1];
    return upper ? (re - im * I) : (re + im * I);
}

/* ---------------------------------------------------------------- real factorisation */

/* Cholesky-Banachiewicz on an n x n real matrix. `l` is a dense n x n column-major scratch
 * (ld = n) that receives L in its lower triangle. Returns info (0 = success). */
static int64_t chol_real(int upper, int64_t n, const double *a, int64_t lda, ldr *l) {
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t j = 0; j < i; ++j) {
            ldr s = in_real(a, lda, upper, i, j);
            for (int64_t k = 0; k < j; ++k) s -= l[k * n + i] * l[k * n + j];
            l[j * n + i] = s / l[j * n + j];
        }
        ldr d = in_real(a, lda, upper, i, i);
        for (int64_t k = 0; k < i; ++k) d -= l[k * n + i] * l[k * n + i];
        if (!(d > 0)) return i + 1;
        l[i * n + i] = sqrtl(d);
    }
    return 0;
}

static int64_t chol_cplx(int upper, int64_t n, const double *a, int64_t lda, ldc *l) {
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t j = 0; j < i; ++j) {
            ldc s = in_cplx(a, lda, upper, i, j);
            for (int64_t k = 0; k < j; ++k) s -= l[k * n + i] * conjl(l[k * n + j]);
            s /= creall(l[j * n + j]);
            l[j * n + i] = s;
        }
        ldr d = creall(in_cplx(a, lda, upper, i, i));
        for (int64_t k = 0; k < i; ++k) {
            ldc v = l[k * n + i];
            d -= creall(v) * creall(v) + cimagl(v) * cimagl(v);
        }
        if (!(d > 0)) return i + 1;
        l[i * n + i] = sqrtl(d);
    }
    return 0;
}

/* ---------------------------------------------------------------- substitutions */

/* Solve L*L^H x = b in place for one right-hand side, L in dense lower storage (ld = n). */
static void solve_real(int64_t n, const ldr *l, ldr *x) {
    for (int64_t i = 0; i < n; ++i) {            /* forward: L*y = b */
        ldr s = x[i];
        for (int64_t k = 0; k < i; ++k) s -= l[k * n + i] * x[k];
        x[i] = s / l[i * n + i];
    }
    for (int64_t i = n - 1; i >= 0; --i) {       /* back: L^H*x = y */
        ldr s = x[i];
        for (int64_t k = i + 1; k < n; ++k) s -= l[i * n + k] * x[k];
        x[i] = s / l[i * n + i];
    }
}

static void solve_cplx(int64_t n, const ldc *l, ldc *x) {
    for (int64_t i = 0; i < n; ++i) {
        ldc s = x[i];
        for (int64_t k = 0; k < i; ++k) s -= l[k * n + i] * x[k];
        x[i] = s / creall(l[i * n + i]);
    }
    for (int64_t i = n - 1; i >= 0; --i) {
        ldc s = x[i];
        for (int64_t k = i + 1; k < n; ++k) s -= conjl(l[i * n + k]) * x[k];
        x[i] = s / creall(l[i * n + i]);
    }
}

/* ---------------------------------------------------------------- one item */

/* Factor one item and, if nrhs > 0 and the factor succeeded, solve.
 * out_f: n x n long double (complex: interleaved) column-major, ld = n; receives the factor in
 *        the referenced triangle (Lower: L; Upper: U = L^H), zeros elsewhere. Only the leading
 *        (info-1) x (info-1) block is meaningful when info > 0.
 * b:     nrhs right-hand sides (ld = ldb, double / interleaved).
 * out_x: n x nrhs long double (ld = n), the solution, or b itself when info > 0.
 * If `factor_given` is nonzero, `a` already holds the factor in its referenced triangle and
 * only the substitutions run (potrs). */
static int64_t one_item(int cplx, int upper, int factor_given, int64_t n, const double *a,
                        int64_t lda, int64_t nrhs, const double *b, int64_t ldb, ldr *out_f,
                        ldr *out_x, void *scratch) {
    int64_t info = 0;
    if (!cplx) {
        ldr *l = (ldr *)scratch;
        memset(l, 0, sizeof(ldr) * (size_t)(n * n));
        if (factor_given) {
            for (int64_t c = 0; c < n; ++c)
                for (int64_t i = c; i < n; ++i) l[c * n + i] = in_real(a, lda, upper, i, c);
        } else {
            info = chol_real(upper, n, a, lda, l);
        }
        if (out_f) {
            memset(out_f, 0, sizeof(ldr) * (size_t)(n * n));
            int64_t m = info ? info - 1 : n;
            for (int64_t c = 0; c < m; ++c)
                for (int64_t i = c; i < m; ++i) {
                    if (upper) out_f[i * n + c] = l[c * n + i];
                    else out_f[c * n + i] = l[c * n + i];
                }
        }
        if (out_x) {
            ldr *x = l + n * n;
            for (int64_t r = 0; r < nrhs; ++r) {
                for (int64_t i = 0; i < n; ++i) x[i] = (ldr)b[r * ldb + i];
                if (!info) solve_real(n, l, x);
                for (int64_t i = 0; i < n; ++i) out_x[r * n + i] = x[i];
            }
        }
    } else {
        ldc *l = (ldc *)scratch;
        for (int64_t t = 0; t < n * n; ++t) l[t] = 0;
        if (factor_given) {
            for (int64_t c = 0; c < n; ++c)
                for (int64_t i = c; i < n; ++i) {
                    ldc v = in_cplx(a, lda, upper, i, c);
                    l[c * n + i] = (i == c) ? (ldc)creall(v) : v;
                }
        } else {
            info = chol_cplx(upper, n, a, lda, l);
        }
        if (out_f) {
            memset(out_f, 0, 2 * sizeof(ldr) * (size_t)(n * n));
            int64_t m = info ? info - 1 : n;
            for (int64_t c = 0; c < m; ++c)
                for (int64_t i = c; i < m; ++i) {
                    ldc v = l[c * n + i];
                    int64_t off = upper ? (i * n + c) : (c * n + i);
                    if (upper) v = conjl(v);
                    out_f[2 * off] = creall(v);
                    out_f[2 * off + 1] = cimagl(v);
                }
        }
        if (out_x) {
            ldc *x = l + n * n;
            for (int64_t r = 0; r < nrhs; ++r) {
                for (int64_t i = 0; i < n; ++i)
                    x[i] = (ldr)b[2 * (r * ldb + i)] + (ldr)b[2 * (r * ldb + i) + 1] * I;
                if (!info) solve_cplx(n, l, x);
                for (int64_t i = 0; i < n; ++i) {
                    out_x[2 * (r * n + i)] = creall(x[i]);
                    out_x[2 * (r * n + i) + 1] = cimagl(x[i]);
                }
            }
        }
    }
    return info;
}

/* ---------------------------------------------------------------- batch, threaded */

typedef struct {
    int cplx, upper, factor_given;
    int64_t n, batch, lda, stride_a, nrhs, ldb, stride_b;
    const double *a, *b;
    ldr *out_f, *out_x;
    int32_t *info;
    int64_t lo, hi;
} job_t;

static void *run_job(void *p) {
    job_t *j = (job_t *)p;
    size_t el = j->cplx ? sizeof(ldc) : sizeof(ldr);
    void *scratch = malloc(el * (size_t)(j->n * j->n + j->n));
    if (!scratch) return (void *)1;
    int64_t sc = j->cplx ? 2 : 1;
    for (int64_t it = j->lo; it < j->hi; ++it) {
        const double *a = j->a + sc * it * j->stride_a;
        const double *b = j->b ? j->b + sc * it * j->stride_b : NULL;
        ldr *of = j->out_f ? j->out_f + sc * it * j->n * j->n : NULL;
        ldr *ox = j->out_x ? j->out_x + sc * it * j->n * j->nrhs : NULL;
        int64_t info = one_item(j->cplx, j->upper, j->factor_given, j->n, a, j->lda, j->nrhs, b,
                                j->ldb, of, ox, scratch);
        if (j->info) j->info[it] = (int32_t)info;
    }
    free(scratch);
    return NULL;
}

/*
 * Batched entry point (the only exported function).
 *   cplx, upper    : 0/1 flags
 *   factor_given   : 0 = potrf (+ posv when nrhs > 0), 1 = potrs (a holds the factor)
 *   a              : input items as doubles (complex: interleaved), ld lda, stride stride_a
 *                    (both in elements)
 *   b              : nrhs right-hand sides per item (ld ldb, stride stride_b), or NULL
 *   out_f          : batch x n x n long double (complex: x2), dense ld = n; or NULL
 *   out_x          : batch x n x nrhs long double (complex: x2), dense ld = n; or NULL
 *   info           : batch int32, or NULL
 *   nthreads       : worker threads (>= 1); items are split into contiguous ranges
 * Returns 0, or -1 when a worker could not allocate its scratch.
 */
int bl_oracle_run(int cplx, int upper, int factor_given, int64_t n, int64_t batch,
                  const double *a, int64_t lda, int64_t stride_a, int64_t nrhs,
                  const double *b, int64_t ldb, int64_t stride_b, long double *out_f,
                  long double *out_x, int32_t *info, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > batch) nthreads = (int)(batch > 0 ? batch : 1);
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        job_t *j = &jobs[t];
        j->cplx = cplx; j->upper = upper; j->factor_given = factor_given;
        j->n = n; j->batch = batch; j->lda = lda; j->stride_a = stride_a;
        j->nrhs = nrhs; j->ldb = ldb; j->stride_b = stride_b;
        j->a = a; j->b = b; j->out_f = out_f; j->out_x = out_x; j->info = info;
        j->lo = batch * t / nthreads; j->hi = batch * (t + 1) / nthreads;
        if (nthreads > 1) {
            if (pthread_create(&th[t], NULL, run_job, j) != 0) { rc = -1; th[t] = 0; }
        } else if (run_job(j) != NULL) {
            rc = -1;
        }
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; ++t) {
            void *ret = NULL;
            if (th[t]) pthread_join(th[t], &ret);
            if (ret != NULL) rc = -1;
        }
    free(jobs); free(th);
    return rc;
}

/* Width of long double in bits of mantissa, so the caller can state which format ran. */
int bl_oracle_ldbl_mant_dig(void) { return __LDBL_MANT_DIG__; }
