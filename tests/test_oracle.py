"""Pins for the CPU oracle: every check compares it with something other than itself.

What fixes each value (BatchLAS "Batched Cholesky (potrf)" page for the semantics):
* integer factors: A = L0*L0^H built exactly from an integer (Gaussian-integer) L0 has the
  exact Cholesky factor L0, so the oracle must return L0 bit for bit;
* closed forms: identity, diagonal, the 2x2 formula;
* info: the first non-positive pivot, 1-based ("potrf: correctness findings" item 6 merges a
  local index as j + leaf; "TinyInfoIsExactAndFirstFailureWins"), pinned by brute-force
  leading minors in exact rational arithmetic and by planted negative and NaN diagonals;
* a third opinion: LAPACK through numpy.linalg on random SPD inputs;
* invariants: residual ||A - L L^H|| near long-double precision, Upper == Lower^H.
"""
import math
from fractions import Fraction
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import synth

LD_EPS = float(np.finfo(np.longdouble).eps)


def _rng(seed):
    return np.random.default_rng(seed)


def _int_factor(rng, n, cplx):
    """Random lower-triangular integer (or Gaussian-integer) factor with positive diagonal."""
    L = np.zeros((n, n), dtype=object)
    for i in range(n):
        for j in range(i):
            re = int(rng.integers(-3, 4))
            L[i, j] = complex(re, int(rng.integers(-3, 4))) if cplx else re
        L[i, i] = int(rng.integers(1, 5))
    return L


def _exact_gram(L, cplx):
    """A = L*L^H in exact Python integer arithmetic."""
    n = L.shape[0]
    A = np.zeros((n, n), dtype=object)
    for i in range(n):
        for j in range(n):
            s = 0
            for k in range(n):
                s += L[i, k] * (L[j, k].conjugate() if cplx else L[j, k])
            A[i, j] = s
    return A


def _to_dtype(A_obj, dtype):
    return np.array(A_obj.tolist(), dtype=synth.DTYPES[dtype])


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("uplo", ["L", "U"])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 12])
def test_integer_factor_is_recovered_exactly(dtype, uplo, n):
    cplx = synth.is_complex(dtype)
    rng = _rng(100 + n)
    L0 = _int_factor(rng, n, cplx)
    A = _exact_gram(L0, cplx)
    assert max(abs(complex(v)) for v in A.flat) < 2 ** 24  # exact in every dtype
    f, info = oracle.potrf(_to_dtype(A, dtype)[None], uplo)
    assert info[0] == 0
    expect = np.array(L0.tolist(), dtype=np.clongdouble if cplx else np.longdouble)
    if uplo == "U":
        expect = np.conj(expect.T)
    assert np.array_equal(f[0], expect), "oracle must reproduce the integer factor bit-exactly"


@pytest.mark.parametrize("dtype", ["f32", "c128"])
def test_identity_and_diagonal(dtype):
    n = 9
    eye = np.eye(n, dtype=synth.DTYPES[dtype])[None]
    for uplo in "LU":
        f, info = oracle.potrf(eye, uplo)
        assert info[0] == 0 and np.array_equal(f[0], np.eye(n))
    squares = np.array([(k + 1) ** 2 for k in range(n)], float)
    D = np.diag(squares).astype(synth.DTYPES[dtype])[None]
    f, info = oracle.potrf(D, "L")
    assert info[0] == 0 and np.array_equal(f[0], np.diag(np.arange(1, n + 1)).astype(np.longdouble))
    # non-square diagonal entries: sqrt correctly rounded to long double
    rng = _rng(5)
    d = rng.uniform(0.5, 50.0, n)
    f, info = oracle.potrf(np.diag(d)[None], "U")
    for k in range(n):
        got = f[0, k, k]
        # |got^2 - d| <= 1 ulp of d at long-double precision (exact rational check)
        g = Fraction(*got.as_integer_ratio())
        err = abs(g * g - Fraction(d[k]))
        assert err <= Fraction(d[k]) * Fraction(LD_EPS) * 2, (k, float(err))
        assert f[0, k, (k + 1) % n] == 0 or n == 1


@pytest.mark.parametrize("cplx", [False, True])
def test_2x2_closed_form(cplx):
    getcontext().prec = 50
    rng = _rng(7)
    for _ in range(20):
        a = float(rng.uniform(1, 10))
        c = float(rng.uniform(5, 20))
        br, bi = float(rng.uniform(-1, 1)), float(rng.uniform(-1, 1)) if cplx else 0.0
        A = np.array([[a, br - 1j * bi], [br + 1j * bi, c]]) if cplx else np.array([[a, br], [br, c]])
        f, info = oracle.potrf(A[None], "L")
        assert info[0] == 0
        sa = Decimal(a).sqrt()
        l21r, l21i = Decimal(br) / sa, Decimal(bi) / sa
        l22 = (Decimal(c) - (Decimal(br) ** 2 + Decimal(bi) ** 2) / Decimal(a)).sqrt()
        tol = 8 * LD_EPS
        assert abs(Decimal(repr(float(f[0, 0, 0].real))) - sa) / sa < Decimal(1e-15)
        got = f[0]
        def close(x, ref):
            return abs(float(x) - float(ref)) <= tol * max(1.0, abs(float(ref))) * 16
        assert close(got[0, 0].real, sa) and close(got[1, 1].real, l22)
        assert close(got[1, 0].real, l21r) and close(got[1, 0].imag if cplx else 0, l21i)
        assert got[0, 1] == 0


def _det_fraction(M):
    """Exact determinant of a square matrix of Fractions / Gaussian rationals (real only)."""
    M = [row[:] for row in M]
    n = len(M)
    det = Fraction(1)
    for c in range(n):
        p = next((r for r in range(c, n) if M[r][c] != 0), None)
        if p is None:
            return Fraction(0)
        if p != c:
            M[c], M[p] = M[p], M[c]
            det = -det
        det *= M[c][c]
        for r in range(c + 1, n):
            f = M[r][c] / M[c][c]
            for k in range(c, n):
                M[r][k] -= f * M[c][k]
    return det


def test_info_matches_brute_force_leading_minors():
    """info = smallest m with det(A[:m,:m]) <= 0 (0 if none), on exact rationals."""
    rng = _rng(11)
    seen = set()
    checked = 0
    for trial in range(400):
        n = int(rng.integers(1, 7))
        X = rng.integers(-4, 5, (n, n)).astype(float)
        A = X @ X.T + np.diag(rng.integers(-6, 7, n).astype(float))
        A = (A + A.T) / 2
        Af = [[Fraction(float(A[i, j])) for j in range(n)] for i in range(n)]
        dets = [Fraction(1)] + [_det_fraction([r[:m] for r in Af[:m]]) for m in range(1, n + 1)]
        # pivots d_m = det_m / det_{m-1} while the leading minors stay positive
        expect, borderline = 0, False
        for m in range(1, n + 1):
            if dets[m - 1] > 0:
                piv = dets[m] / dets[m - 1]
                if abs(piv) < Fraction(1, 1000) * (1 + abs(Af[m - 1][m - 1])):
                    borderline = True
            if dets[m] <= 0:
                expect = m
                break
        if borderline:
            continue
        for uplo in "LU":
            _, info = oracle.potrf(A[None], uplo)
            assert info[0] == expect, (A, expect, info[0])
        seen.add(expect)
        checked += 1
    assert checked > 200 and len(seen) >= 5, (checked, seen)


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_planted_failures(dtype):
    rng = _rng(13)
    n = 10
    A = synth.spd_bbt(rng, n, 6, dtype)
    A[0, 0, 0] = -1              # info 1
    A[1, 4, 4] = -1              # info 5
    A[2, 9, 9] = np.nan          # info 10, NaN pivot
    A[3, 2, 2] = -1
    A[3, 6, 6] = -1              # two planted: the smaller wins -> 3
    A[4, 7, 7] = 0               # the pivot is negative once the Schur update applies -> 8
    expect = [1, 5, 10, 3, 8, 0]
    for uplo in "LU":
        f, info = oracle.potrf(A, uplo)
        assert list(info) == expect
        # the factor's leading block still matches the factor of the leading block
        f2, info2 = oracle.potrf(A[1:2, :4, :4].copy(), uplo)
        assert info2[0] == 0
        assert np.array_equal(f[1, :4, :4], f2[0])


@pytest.mark.parametrize("dtype", ["f64", "c128"])
@pytest.mark.parametrize("kind", ["bbt", "haar"])
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_lapack_third_opinion(dtype, kind, uplo):
    rng = _rng(17)
    n = 24
    gen = synth.spd_bbt if kind == "bbt" else synth.spd_haar
    A = gen(rng, n, 8, dtype)
    f, info = oracle.potrf(A, uplo)
    assert not info.any()
    ref = np.linalg.cholesky(A)
    if uplo == "U":
        ref = np.conj(np.swapaxes(ref, -1, -2))
    wide = np.complex128 if synth.is_complex(dtype) else np.float64
    for b in range(A.shape[0]):
        kappa = np.linalg.cond(A[b])
        err = np.linalg.norm(f[b].astype(wide) - ref[b]) / np.linalg.norm(ref[b])
        assert err <= n * kappa * 1e-15, (b, err, kappa)


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_residual_at_long_double_precision(dtype):
    rng = _rng(19)
    n = 20
    A = synth.spd_bbt(rng, n, 4, dtype)
    for uplo in "LU":
        f, info = oracle.potrf(A, uplo)
        assert not info.any()
        Aw = A.astype(np.clongdouble if synth.is_complex(dtype) else np.longdouble)
        for b in range(A.shape[0]):
            F = f[b]
            prod = F @ np.conj(F.T) if uplo == "L" else np.conj(F.T) @ F
            res = np.sqrt(np.sum(np.abs(Aw[b] - prod) ** 2)) / np.sqrt(np.sum(np.abs(Aw[b]) ** 2))
            assert res <= 8 * n * LD_EPS, (b, float(res))


def test_upper_is_lower_conjugate_transpose():
    rng = _rng(23)
    for dtype in ("f64", "c128"):
        A = synth.spd_bbt(rng, 15, 3, dtype)
        fl, il = oracle.potrf(A, "L")
        fu, iu = oracle.potrf(A, "U")
        assert not il.any() and not iu.any()
        assert np.array_equal(fu, np.conj(np.swapaxes(fl, -1, -2)))


def test_upper_reads_only_its_triangle():
    """Poisoning the unreferenced triangle with NaN changes nothing."""
    rng = _rng(29)
    A = synth.spd_bbt(rng, 11, 2, "c128")
    for uplo in "LU":
        P = A.copy()
        iu = np.triu_indices(11, 1) if uplo == "L" else np.tril_indices(11, -1)
        P[:, iu[0], iu[1]] = np.nan
        f0, i0 = oracle.potrf(A, uplo)
        f1, i1 = oracle.potrf(P, uplo)
        assert np.array_equal(f0, f1) and np.array_equal(i0, i1)


@pytest.mark.parametrize("cplx", [False, True])
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_posv_integer_solution_is_exact(cplx, uplo):
    """With an integer factor L0 and integer X0, B = L0 L0^H X0 is exact and every
    substitution step divides exactly, so X must equal X0 bit for bit."""
    rng = _rng(31)
    n, nrhs = 9, 3
    L0 = _int_factor(rng, n, cplx)
    A = _exact_gram(L0, cplx)
    X0 = np.zeros((n, nrhs), dtype=object)
    for i in range(n):
        for r in range(nrhs):
            re = int(rng.integers(-5, 6))
            X0[i, r] = complex(re, int(rng.integers(-5, 6))) if cplx else re
    B = np.zeros((n, nrhs), dtype=object)
    for i in range(n):
        for r in range(nrhs):
            B[i, r] = sum(A[i, k] * X0[k, r] for k in range(n))
    dt = "c128" if cplx else "f64"
    f, x, info = oracle.posv(_to_dtype(A, dt)[None], _to_dtype(B, dt)[None], uplo)
    assert info[0] == 0
    expect = np.array(X0.tolist(), dtype=np.clongdouble if cplx else np.longdouble)
    assert np.array_equal(x[0], expect)
    # potrs with the exact factor gives the same exact solution
    F = np.array(L0.tolist(), dtype=synth.DTYPES[dt])
    if uplo == "U":
        F = np.conj(F.T)
    xs = oracle.potrs(F[None], _to_dtype(B, dt)[None], uplo)
    assert np.array_equal(xs[0], expect)


def test_posv_closed_forms_and_failure():
    rng = _rng(37)
    n, nrhs = 7, 4
    B = synth.rhs_uniform(rng, n, nrhs, 1, "f64")
    _, x, info = oracle.posv(np.eye(n)[None], B, "L")
    assert info[0] == 0 and np.array_equal(x[0], B[0].astype(np.longdouble))
    d = np.array([4.0, 16.0, 64.0, 0.25, 0.0625, 256.0, 1.0])  # squares of powers of two
    _, x, info = oracle.posv(np.diag(d)[None], B, "U")
    assert np.array_equal(x[0], (B[0] / d[:, None]).astype(np.longdouble))
    # failure leaves B unchanged
    A = synth.spd_bbt(rng, n, 1, "f64")
    A[0, 3, 3] = -1
    _, x, info = oracle.posv(A, B, "L")
    assert info[0] == 4 and np.array_equal(x[0], B[0].astype(np.longdouble))


@pytest.mark.parametrize("dtype", ["f64", "c128"])
def test_posv_lapack_third_opinion(dtype):
    rng = _rng(41)
    n, nrhs = 30, 5
    A = synth.spd_haar(rng, n, 4, dtype)
    B = synth.rhs_uniform(rng, n, nrhs, 4, dtype)
    for uplo in "LU":
        _, x, info = oracle.posv(A, B, uplo)
        assert not info.any()
        ref = np.linalg.solve(A, B)
        wide = np.complex128 if synth.is_complex(dtype) else np.float64
        for b in range(4):
            err = np.linalg.norm(x[b].astype(wide) - ref[b]) / np.linalg.norm(ref[b])
            assert err <= n * np.linalg.cond(A[b]) * 1e-15


def test_non_natural_layout_matches_natural():
    """ld = n+7 and stride = ld*n+13 read the same matrices (the gaps are poisoned)."""
    rng = _rng(43)
    n, batch = 13, 3
    A = synth.spd_bbt(rng, n, batch, "c64")
    ld, stride = n + 7, (n + 7) * n + 13
    buf = synth.to_colmajor(A, ld, stride, fill=np.nan)
    f1, _, i1 = oracle.run("L", n, batch, buf, ld, stride)
    f0, i0 = oracle.potrf(A, "L")
    assert np.array_equal(f0, f1) and np.array_equal(i0, i1)


def test_threads_do_not_change_results():
    rng = _rng(47)
    A = synth.spd_bbt(rng, 16, 37, "f32")
    f1, i1 = oracle.potrf(A, "U", threads=1)
    f4, i4 = oracle.potrf(A, "U", threads=4)
    assert np.array_equal(f1, f4) and np.array_equal(i1, i4)


def test_layout_roundtrip():
    rng = _rng(53)
    A = synth.spd_bbt(rng, 5, 4, "c128")
    buf = synth.to_colmajor(A, 8, 8 * 5 + 3)
    assert np.array_equal(synth.from_colmajor(buf, 5, 5, 4, 8, 43), A)
    # element (i, j) of item b sits at b*stride + j*ld + i
    assert buf[2 * 43 + 3 * 8 + 1] == A[2, 1, 3]
