"""Hand-derived worked examples (tests/golden/worked_examples.txt): each A = L0 L0^H with an
integer or Gaussian-integer L0, so the exact factor is L0 and, with B = A X0, the exact
solution is X0; failure cases give the exact 1-based first failing pivot. The derivations and
the passages they follow are written next to each case in the fixture file.

The oracle must reproduce every value exactly (integer data stays exact in long double); the
library, through its C ABI, within the stated tolerances, for every compiled route pinned in
turn, Lower and Upper, on a batch of copies that leaves a ragged last group.
"""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _rows(text, cplx):
    conv = complex if cplx else int
    return [[conv(t) for t in r.split()] for r in text.split(";")]


def load_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest, "cite": None}
            elif key == "cite":
                cur["cite"] = rest
            elif key in ("A", "L", "X", "B"):
                cur[key] = rest
            elif key == "info":
                cur["info"] = int(rest)
            elif key == "end":
                cplx = any("j" in cur.get(k, "") for k in ("A", "L", "X", "B"))
                cur["cplx"] = cplx
                for k in ("A", "L", "X", "B"):
                    if k in cur:
                        cur[k] = np.array(_rows(cur[k], cplx), dtype=object)
                cases.append(cur)
                cur = None
    return cases


CASES = load_cases()
IDS = [c["name"] for c in CASES]


def test_fixture_file_is_complete():
    assert len(CASES) >= 9
    for c in CASES:
        assert c["cite"], c["name"]
        n = c["A"].shape[0]
        assert c["A"].shape == (n, n)
        if c["info"] == 0:
            assert c["L"].shape == (n, n)
        elif "L" in c:
            assert c["L"].shape == (c["info"] - 1, c["info"] - 1)


def test_fixtures_are_consistent_by_exact_arithmetic():
    """The fixture's own claims hold in exact integer arithmetic: A = L L^H on the referenced
    block, B = A X."""
    for c in CASES:
        A, cplx = c["A"], c["cplx"]
        if "L" in c:
            L = c["L"]
            m = L.shape[0]
            LH = np.array([[x.conjugate() if cplx else x for x in row] for row in L.T], dtype=object)
            prod = L.dot(LH)
            for i in range(m):
                for j in range(m):
                    a = A[i, j]
                    if i == j and cplx:
                        a = complex(a.real, 0)                 # the diagonal's imaginary part is ignored
                    assert prod[i, j] == a, (c["name"], i, j)
        if "X" in c:
            assert (A if not any(isinstance(x, complex) and x.imag for x in np.diag(A)) else
                    _hermitian_part(A)).dot(c["X"]).tolist() == c["B"].tolist(), c["name"]


def _hermitian_part(A):
    H = A.copy()
    for i in range(A.shape[0]):
        H[i, i] = complex(A[i, i].real, 0)
    return H


def _dtypes(c):
    return ["c64", "c128"] if c["cplx"] else ["f32", "f64", "c64", "c128"]


def _logical(M, dtype, copies):
    return np.repeat(np.array(M.tolist(), dtype=synth.DTYPES[dtype])[None], copies, axis=0)


def _exact_dtype(c, dtype):
    return np.complex128 if (c["cplx"] or synth.is_complex(dtype)) else np.float64


def _expected_factor(c, uplo, dtype):
    L = np.array(c["L"].tolist(), dtype=_exact_dtype(c, dtype))
    return L if uplo == "L" else np.conj(L.T)


@pytest.mark.parametrize("c", CASES, ids=IDS)
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_oracle_reproduces_worked_examples_exactly(c, uplo):
    n = c["A"].shape[0]
    for dtype in _dtypes(c):
        A = _logical(c["A"], dtype, 1)
        buf = synth.to_colmajor(A)
        nrhs = c["X"].shape[1] if "X" in c else 0
        bbuf = synth.to_colmajor(_logical(c["B"], dtype, 1)) if nrhs else None
        F, X, info = oracle.run(uplo, n, 1, buf, n, n * n, nrhs, bbuf, n, n * nrhs)
        assert info[0] == c["info"], (c["name"], dtype)
        if "L" in c:
            m = c["L"].shape[0]
            exp = _expected_factor(c, uplo, dtype)
            got = F[0][:m, :m]
            assert np.array_equal(got.astype(exp.dtype), exp), (c["name"], dtype, uplo)
        if nrhs and c["info"] == 0:
            exp = np.array(c["X"].tolist(), dtype=_exact_dtype(c, dtype))
            assert np.array_equal(X[0].astype(exp.dtype), exp), (c["name"], dtype, uplo)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_library_reproduces_worked_examples_on_every_route(dtype):
    from _gpu import TOL_F, TOL_X, call_posv, call_potrf, lib
    bl = lib()
    copies = 37
    for spelling, cap, rhs in bl.routes(dtype):
        for c in CASES:
            if dtype not in _dtypes(c):
                continue
            n = c["A"].shape[0]
            if cap and n > cap:
                continue
            for uplo in ("L", "U"):
                A = _logical(c["A"], dtype, copies)
                _, out, info, _, _ = call_potrf(A, uplo, dtype, route=spelling)
                assert (info == c["info"]).all(), (spelling, c["name"], uplo, info[:4])
                if "L" in c:
                    m = c["L"].shape[0]
                    F = synth.from_colmajor(out, n, n, copies)
                    exp = _expected_factor(c, uplo, dtype)
                    mask = np.tril(np.ones((m, m), bool)) if uplo == "L" else np.triu(np.ones((m, m), bool))
                    for b in (0, copies - 1):
                        g = np.where(mask, F[b][:m, :m], 0).astype(exp.dtype)
                        err = np.linalg.norm(g - exp) / np.linalg.norm(exp)
                        assert err <= TOL_F[dtype], (spelling, c["name"], uplo, err)
                if "X" in c and rhs >= 0 and (rhs == 0 or rhs >= c["X"].shape[1]) and c["info"] == 0:
                    B = _logical(c["B"], dtype, copies)
                    _, _, _, bout, pinfo = call_posv(A, B, uplo, dtype, route=spelling)
                    assert (pinfo == 0).all(), (spelling, c["name"], uplo)
                    X = synth.from_colmajor(bout, n, c["X"].shape[1], copies)
                    exp = np.array(c["X"].tolist(), dtype=_exact_dtype(c, dtype))
                    for b in (0, copies - 1):
                        err = np.linalg.norm(X[b].astype(exp.dtype) - exp) / np.linalg.norm(exp)
                        assert err <= TOL_X[dtype], (spelling, c["name"], uplo, err)
