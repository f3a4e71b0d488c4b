"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Every case calls the library through its C ABI (libbl.so) and compares element by element
with the oracle (BatchLAS "Batched Cholesky (potrf)" page for the semantics: info is the
1-based first failing pivot, bit-exact; the factor within the stated tolerance; the other
triangle neither read nor written).
"""
import numpy as np
import pytest

import oracle
import synth
from _gpu import (TOL_F, TOL_X, THREADS, call_posv, call_potrf, factor_errors, lib,
                  other_triangle_unchanged, solution_errors, torch_cuda)

pytestmark = pytest.mark.gpu

# (workload, reduced batch for the all-items comparison)
SMALL = [("f32_n8", None), ("f32_n32", 1024), ("f64_n17", 512), ("f64_n33", 256), ("f64_n65", 128),
         ("c64_n128", 24), ("f32_n512", 2), ("f64_n512", 2)]


def _check_potrf(A, uplo, dtype, expect_info=None, **kw):
    in_buf, out_buf, info, ld, stride = call_potrf(A, uplo, dtype, **kw)
    batch, n, _ = A.shape
    ref, _, rinfo = oracle.run(uplo, n, batch, in_buf, ld, stride, threads=THREADS)
    assert np.array_equal(info, rinfo), f"info mismatch at {np.nonzero(info != rinfo)[0][:10]}"
    if expect_info is not None:
        assert np.array_equal(info, expect_info)
    errs = factor_errors(out_buf, ref, info, n, batch, ld, stride, uplo)
    assert errs.max() <= TOL_F[dtype], f"max factor error {errs.max():.3e} (item {errs.argmax()})"
    assert other_triangle_unchanged(in_buf, out_buf, n, batch, ld, stride, uplo)
    return out_buf, info, errs


@pytest.mark.parametrize("name,batch", SMALL, ids=[s[0] for s in SMALL])
def test_potrf_workloads_all_items(name, batch):
    w = synth.workload(name, batch)
    for uplo in ("L", "U"):
        _check_potrf(w.A, uplo, w.dtype, expect_info=w.planted_info)


@pytest.mark.parametrize("name,batch", [("f32_n32", 512), ("c64_n128", 16), ("f64_n512", 2)])
def test_posv_workloads_all_items(name, batch):
    w = synth.workload(name, batch)
    for uplo in ("L", "U"):
        abuf, aout, bbuf, bout, info = call_posv(w.A, w.B, uplo, w.dtype)
        n, nrhs, b = w.n, w.nrhs, w.batch
        ref, x, rinfo = oracle.run(uplo, n, b, abuf, n, n * n, nrhs, bbuf, n, n * nrhs, threads=THREADS)
        assert np.array_equal(info, rinfo) and not info.any()
        assert factor_errors(aout, ref, info, n, b, n, n * n, uplo).max() <= TOL_F[w.dtype]
        X = synth.from_colmajor(bout, n, nrhs, b)
        e = solution_errors(X, x)
        assert e.max() <= TOL_X[w.dtype], f"max solution error {e.max():.3e}"


FULL = ["f32_n8", "f32_n32", "f64_n17", "f64_n33", "f64_n65", "c64_n128", "f32_n512", "f64_n512"]


@pytest.mark.parametrize("name", FULL)
def test_potrf_full_size_sampled(name):
    """The full workload in one launch (as the benchmark runs it); the oracle checks a sample
    of items, the first and last included; info is checked for every item."""
    w = synth.workload(name)
    nsamp = 3 if w.n >= 512 else 24
    items = np.unique(np.linspace(0, w.batch - 1, nsamp).astype(int))
    for uplo in w.uplos:
        in_buf, out_buf, info, ld, stride = call_potrf(w.A, uplo, w.dtype)
        expect = w.planted_info if w.planted_info is not None else np.zeros(w.batch, np.int32)
        assert np.array_equal(info, expect)
        sub = synth.to_colmajor(w.A[items])
        ref, _, rinfo = oracle.run(uplo, w.n, len(items), sub, w.n, w.n * w.n, threads=THREADS)
        assert np.array_equal(rinfo, info[items])
        errs = factor_errors(out_buf, ref, info, w.n, w.batch, ld, stride, uplo, items=items)
        assert errs.max() <= TOL_F[w.dtype], f"{name} {uplo}: {errs.max():.3e}"


@pytest.mark.parametrize("name", ["f32_n32", "c64_n128", "f64_n512"])
def test_posv_full_size_sampled(name):
    w = synth.workload(name)
    nsamp = 3 if w.n >= 512 else 16
    items = np.unique(np.linspace(0, w.batch - 1, nsamp).astype(int))
    abuf, aout, bbuf, bout, info = call_posv(w.A, w.B, "L", w.dtype)
    assert not info.any()
    _, x, _ = oracle.run("L", w.n, len(items), synth.to_colmajor(w.A[items]), w.n, w.n * w.n, w.nrhs,
                         synth.to_colmajor(w.B[items]), w.n, w.n * w.nrhs, want_factor=False, threads=THREADS)
    X = synth.from_colmajor(bout, w.n, w.nrhs, w.batch)[items]
    assert solution_errors(X, x).max() <= TOL_X[w.dtype]


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_every_route_pinned_at_its_capacity(dtype):
    """Each compiled variant runs at the largest order it admits and refuses one more
    (can_run equals what the launch accepts)."""
    bl = lib()
    rng = np.random.default_rng(3)
    for spelling, cap, rhs in bl.routes(dtype):
        ns = [cap, max(1, cap - 5)] if cap else [1, 37, 200]
        for n in ns:
            A = synth.spd_bbt(rng, n, 5 if n < 300 else 2, dtype)
            _check_potrf(A, "L", dtype, route=spelling)
            _check_potrf(A, "U", dtype, route=spelling)
        if cap:
            A = synth.spd_bbt(rng, cap + 1, 1, dtype)
            with pytest.raises(bl.BLError) as e:
                call_potrf(A, "L", dtype, route=spelling)
            assert e.value.status == 1


@pytest.mark.parametrize("dtype", ["f32", "c128"])
def test_every_route_pinned_posv_and_potrs(dtype):
    bl = lib()
    rng = np.random.default_rng(5)
    for spelling, cap, rhs in bl.routes(dtype):
        if rhs < 0:        # factor-only variant
            continue
        any_rhs = rhs == 0                       # blocked variants take any number per pass
        n = (cap - (0 if any_rhs else min(rhs, 3))) if cap else 70
        n = min(n, 300)
        nrhs = 3 if (any_rhs or rhs >= 3) else rhs
        if n < 1:
            continue
        A = synth.spd_bbt(rng, n, 3, dtype)
        B = synth.rhs_uniform(rng, n, nrhs, 3, dtype)
        for uplo in "LU":
            abuf, aout, bbuf, bout, info = call_posv(A, B, uplo, dtype, route=spelling)
            _, x, rinfo = oracle.run(uplo, n, 3, abuf, n, n * n, nrhs, bbuf, n, n * nrhs, threads=THREADS)
            assert not info.any()
            assert solution_errors(synth.from_colmajor(bout, n, nrhs, 3), x).max() <= TOL_X[dtype], spelling
            # potrs on the oracle's factor rounded to the dtype
            F, _, _ = oracle.run(uplo, n, 3, abuf, n, n * n, threads=THREADS)
            Fd = F.astype(np.complex128 if synth.is_complex(dtype) else np.float64).astype(synth.DTYPES[dtype])
            fbuf = synth.to_colmajor(Fd)
            xs = oracle.run(uplo, n, 3, fbuf, n, n * n, nrhs, bbuf, n, n * nrhs, factor_given=True,
                            want_factor=False, threads=THREADS)[1]
            _, _, _, bout2, _ = call_posv(Fd, B, uplo, dtype, route=spelling, op="potrs")
            assert solution_errors(synth.from_colmajor(bout2, n, nrhs, 3), xs).max() <= TOL_X[dtype], spelling


def test_posv_many_rhs_runs_in_passes():
    """nrhs above the fused kernel's per-pass limit runs further solve-only passes; a failed
    item's right-hand sides stay untouched in every pass."""
    rng = np.random.default_rng(7)
    n, nrhs, batch = 20, 13, 9
    A = synth.spd_bbt(rng, n, batch, "f32")
    A[4, 6, 6] = -1
    B = synth.rhs_uniform(rng, n, nrhs, batch, "f32")
    for route in ("tile:p=4:s=6", "tile:p=8:s=5", "blocked:nb=32"):
        abuf, aout, bbuf, bout, info = call_posv(A, B, "L", "f32", route=route)
        _, x, rinfo = oracle.run("L", n, batch, abuf, n, n * n, nrhs, bbuf, n, n * nrhs, threads=THREADS)
        assert np.array_equal(info, rinfo) and info[4] == 7
        X = synth.from_colmajor(bout, n, nrhs, batch)
        ok = np.arange(batch) != 4
        assert solution_errors(X[ok], x[ok]).max() <= TOL_X["f32"]
        assert np.array_equal(np.ascontiguousarray(X[4]).view(np.uint8), np.ascontiguousarray(B[4]).view(np.uint8)), route


@pytest.mark.parametrize("dtype", ["f32", "c64", "f64"])
def test_non_natural_layout_is_bit_identical(dtype):
    """ld = n+7, stride = ld*n+13 with NaN in every gap: same bits as the natural layout."""
    rng = np.random.default_rng(11)
    for n in (7, 32, 65, 130):
        if n > 100 and dtype == "f64":
            continue
        A = synth.spd_bbt(rng, n, 6, dtype)
        for uplo in "LU":
            _, o0, i0, ld0, s0 = call_potrf(A, uplo, dtype)
            ld, st = n + 7, (n + 7) * n + 13
            in1, o1, i1, _, _ = call_potrf(A, uplo, dtype, ld=ld, stride=st, fill=np.nan)
            f0 = synth.from_colmajor(o0, n, n, 6, ld0, s0)
            f1 = synth.from_colmajor(o1, n, n, 6, ld, st)
            m = np.broadcast_to(np.tril(np.ones((n, n), bool)) if uplo == "L" else np.triu(np.ones((n, n), bool)), f0.shape)
            assert np.array_equal(np.ascontiguousarray(f0[m]).view(np.uint8),
                                  np.ascontiguousarray(f1[m]).view(np.uint8))
            assert np.array_equal(i0, i1)
            assert other_triangle_unchanged(in1, o1, n, 6, ld, st, uplo)


@pytest.mark.parametrize("dtype", ["f32", "c128"])
def test_other_triangle_is_neither_read_nor_written(dtype):
    """NaN in the other triangle changes no bit of the result (not read); a finite sentinel
    there survives bit-exactly (not written)."""
    rng = np.random.default_rng(13)
    for n in (5, 32, 100):
        A = synth.spd_bbt(rng, n, 4, dtype)
        for uplo in "LU":
            other = ~(np.tril(np.ones((n, n), bool)) if uplo == "L" else np.triu(np.ones((n, n), bool)))
            P = A.copy()
            P[:, other] = np.nan
            S = A.copy()
            S[:, other] = (-999 + 777j) if synth.is_complex(dtype) else -999
            _, o0, i0, _, _ = call_potrf(A, uplo, dtype)
            _, o1, i1, _, _ = call_potrf(P, uplo, dtype)
            in2, o2, i2, _, _ = call_potrf(S, uplo, dtype)
            tri = ~other
            f0, f1 = synth.from_colmajor(o0, n, n, 4), synth.from_colmajor(o1, n, n, 4)
            assert np.array_equal(np.ascontiguousarray(f0[:, tri]).view(np.uint8),
                                  np.ascontiguousarray(f1[:, tri]).view(np.uint8))
            assert np.array_equal(i0, i1) and not i1.any()
            assert other_triangle_unchanged(in2, o2, n, 4, n, n * n, uplo)


def test_saturating_identical_batch_is_bit_identical():
    """2048 copies of one matrix give 2048 bit-identical factors, equal to the solo run
    (packed == solo; a race would show only at saturating occupancy)."""
    rng = np.random.default_rng(17)
    for dtype, n in (("f32", 32), ("f32", 8), ("c64", 128), ("f64", 65), ("f32", 300)):
        one = synth.spd_bbt(rng, n, 1, dtype)
        batch = 2048 if n <= 128 else 160
        A = np.repeat(one, batch, axis=0)
        _, o, info, _, _ = call_potrf(A, "L", dtype)
        F = synth.from_colmajor(o, n, n, batch)
        assert not info.any()
        assert np.array_equal(F, np.broadcast_to(F[:1], F.shape)), (dtype, n)
        _, o1, _, _, _ = call_potrf(one, "L", dtype)
        assert np.array_equal(synth.from_colmajor(o1, n, n, 1), F[:1])


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_planted_failures_report_the_first_pivot(dtype):
    rng = np.random.default_rng(19)
    for n in (6, 17, 40, 129, 300):
        if dtype == "c128" and n > 130:
            continue
        A = synth.spd_bbt(rng, n, 6, dtype)
        A[0, 0, 0] = -1
        A[1, n - 1, n - 1] = -1
        A[2, n // 2, n // 2] = np.nan
        A[3, n // 3, n // 3] = -1
        A[3, n // 2 + 1, n // 2 + 1] = -1
        expect = np.array([1, n, n // 2 + 1, n // 3 + 1, 0, 0], np.int32)
        for uplo in "LU":
            _check_potrf(A, uplo, dtype, expect_info=expect)
        B = synth.rhs_uniform(rng, n, 2, 6, dtype)
        abuf, aout, bbuf, bout, info = call_posv(A, B, "L", dtype)
        assert np.array_equal(info, expect)
        Xg = synth.from_colmajor(bout, n, 2, 6)
        for b in range(4):  # failed items keep their right-hand sides bit for bit
            assert np.array_equal(np.ascontiguousarray(Xg[b]).view(np.uint8), np.ascontiguousarray(B[b]).view(np.uint8))


def test_edge_cases_and_argument_errors():
    torch = torch_cuda()
    bl = lib()
    rng = np.random.default_rng(23)
    # n = 1, batch = 1, ragged batches around the per-CTA packing
    for n, batch in ((1, 1), (1, 33), (2, 1), (3, 7), (8, 9), (16, 17), (33, 3), (144, 1), (161, 2)):
        A = synth.spd_bbt(rng, n, batch, "f32")
        _check_potrf(A, "L", "f32")
        _check_potrf(A, "U", "f32")
    d = torch.zeros(64, device="cuda")
    info = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    bad = [
        lambda: bl.potrf_ptr("L", bl.BL_F32, 0, 1, d.data_ptr(), 1, 1, info.data_ptr(), s),        # n = 0
        lambda: bl.potrf_ptr("L", bl.BL_F32, 4, 0, d.data_ptr(), 4, 16, info.data_ptr(), s),       # batch = 0
        lambda: bl.potrf_ptr("L", bl.BL_F32, 4, 1, d.data_ptr(), 3, 16, info.data_ptr(), s),       # lda < n
        lambda: bl.potrf_ptr("L", bl.BL_F32, 4, 2, d.data_ptr(), 4, 15, info.data_ptr(), s),       # overlap
        lambda: bl.potrf_ptr("L", bl.BL_F32, 4, 1, 0, 4, 16, info.data_ptr(), s),                  # A NULL
        lambda: bl.potrf_ptr("L", bl.BL_F32, 4, 1, d.data_ptr(), 4, 16, 0, s),                     # info NULL
        lambda: bl.potrf_ptr("L", 9, 4, 1, d.data_ptr(), 4, 16, info.data_ptr(), s),               # dtype
        lambda: bl.posv_ptr("L", bl.BL_F32, 4, 0, 1, d.data_ptr(), 4, 16, d.data_ptr(), 4, 4, info.data_ptr(), s),
        lambda: bl.posv_ptr("L", bl.BL_F32, 4, 2, 1, d.data_ptr(), 4, 16, d.data_ptr(), 3, 8, info.data_ptr(), s),
    ]
    for f in bad:
        with pytest.raises(bl.BLError) as e:
            f()
        assert e.value.status == 1
    for spelling in ("tile:p=3:s=3", "nonsense", "tile:p=2:s=2"):
        bl.set_route("potrf", spelling)
        try:
            with pytest.raises(bl.BLError):
                bl.potrf_ptr("L", bl.BL_F32, 9, 1, d.data_ptr(), 9, 81, info.data_ptr(), s)
        finally:
            bl.set_route("potrf", None)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", ["f64", "c128"])
def test_lane_pair_thread_routes_are_bit_identical(dtype):
    """thread:n=N:p=2 (two lanes per matrix, each summing one parity of k, added in the same
    order) gives the bits and info of thread:n=N, and thread:n=N:e=1 (fully unrolled at n = N)
    those of the row loop, also with failing pivots at odd and even columns and a NaN, for Lower
    and Upper and orders below the capacity."""
    bl = lib()
    rng = np.random.default_rng(41)
    routes = {sp: cap for sp, cap, _ in bl.routes(dtype)}
    general = max((c, r) for r, c in routes.items() if r.startswith("thread:") and ":" not in r[7:])[1]
    for sp, cap in routes.items():
        if not sp.startswith("thread:") or (":p=2" not in sp and ":e=1" not in sp):
            continue
        # the unrolled order-N path against the row loop of the widest one-lane route
        base = sp.replace(":p=2", "") if ":p=2" in sp else general
        assert base in routes, base
        for n in sorted({cap, cap - 1, max(1, cap - 6)}):
            A = synth.spd_bbt(rng, n, 131, dtype)
            A[3, n - 1, n - 1] = -1.0
            A[4, n // 2, n // 2] = -1.0
            A[5, (n - 1) // 3, (n - 1) // 3] = np.nan
            for uplo in "LU":
                o0, i0, _ = _check_potrf(A, uplo, dtype, route=base)
                o1, i1, _ = _check_potrf(A, uplo, dtype, route=sp)
                assert np.array_equal(i0, i1), (sp, n, uplo)
                f0, f1 = synth.from_colmajor(o0, n, n, 131), synth.from_colmajor(o1, n, n, 131)
                ok = i0 == 0
                assert np.array_equal(np.ascontiguousarray(f0[ok]).view(np.uint8),
                                      np.ascontiguousarray(f1[ok]).view(np.uint8)), (sp, n, uplo)


def test_pair_row_routes_leave_the_other_triangle():
    """Every float2-pair-row route, pinned: NaN in the other triangle changes no bit of the
    factor (its slab copy and pick read only the referenced triangle's values into the factor)
    and a sentinel there survives (the Upper store writes column i of U only in rows <= i)."""
    bl = lib()
    rng = np.random.default_rng(31)
    for sp, n, _ in bl.routes("f32"):
        if ":v2=1" not in sp:
            continue
        A = synth.spd_bbt(rng, n, 37, "f32")
        for uplo in "LU":
            other = ~(np.tril(np.ones((n, n), bool)) if uplo == "L" else np.triu(np.ones((n, n), bool)))
            P = A.copy()
            P[:, other] = np.nan
            S = A.copy()
            S[:, other] = -999
            _, o0, i0, _, _ = call_potrf(A, uplo, "f32", route=sp)
            _, o1, i1, _, _ = call_potrf(P, uplo, "f32", route=sp)
            in2, o2, i2, _, _ = call_potrf(S, uplo, "f32", route=sp)
            tri = ~other
            f0, f1 = synth.from_colmajor(o0, n, n, 37), synth.from_colmajor(o1, n, n, 37)
            assert np.array_equal(np.ascontiguousarray(f0[:, tri]).view(np.uint8),
                                  np.ascontiguousarray(f1[:, tri]).view(np.uint8)), (sp, uplo)
            assert not i0.any() and not i1.any() and not i2.any(), (sp, uplo)
            assert other_triangle_unchanged(in2, o2, n, 37, n, n * n, uplo), (sp, uplo)


def test_upper_equals_lower_transposed_bitwise_for_real_types():
    """Upper is a load/store transform of the same recurrence: for real types the Upper factor
    is bit-identical to the transposed Lower factor."""
    rng = np.random.default_rng(29)
    bl = lib()
    for n in (8, 32, 100, 200, 300):
        A = synth.spd_bbt(rng, n, 4, "f32")
        _, ol, _, _, _ = call_potrf(A, "L", "f32")
        route = bl.last_choice()                  # the tables may pick different kernels per uplo
        _, ou, _, _, _ = call_potrf(A, "U", "f32", route=route)
        L = synth.from_colmajor(ol, n, n, 4)
        U = synth.from_colmajor(ou, n, n, 4)
        low = np.tril(np.ones((n, n), bool))
        assert np.array_equal(L[:, low], np.swapaxes(U, -1, -2)[:, low]), n


def test_look_ahead_and_pair_rows_are_bit_identical():
    """The look-ahead variants (warp:...:la=1) form the next pivot on its owner lane with the
    same fused multiply-add the rank-1 update applies, and the float2-pair-row variants
    (warp:...:v2=1) apply the same operations in the same order as the packed variant: identical
    bits and info to the plain packed variant, failures included."""
    bl = lib()
    rng = np.random.default_rng(23)
    routes = {sp: cap for sp, cap, _ in bl.routes("f32")}
    for sp, n in routes.items():
        if ":la=1" not in sp and ":v2=1" not in sp:
            continue
        base = sp.replace(":la=1", "").replace(":v2=1", "")
        assert base in routes, base
        A = synth.spd_bbt(rng, n, 3001, "f32")
        A[7, 0, 0] = -1.0
        A[8, n - 1, n - 1] = -1.0
        A[9, n // 2, n // 2] = np.nan
        for uplo in "LU":
            o0, i0, _ = _check_potrf(A, uplo, "f32", route=base)
            o1, i1, _ = _check_potrf(A, uplo, "f32", route=sp)
            assert np.array_equal(i0, i1)
            f0, f1 = synth.from_colmajor(o0, n, n, 3001), synth.from_colmajor(o1, n, n, 3001)
            ok = i0 == 0
            assert np.array_equal(np.ascontiguousarray(f0[ok]).view(np.uint8), np.ascontiguousarray(f1[ok]).view(np.uint8)), sp


def test_pair_row_solve_is_bit_identical():
    """posv on the float2-pair-row variants (fused solve, look-ahead pivots) gives the same bits
    in A and B and the same info as the packed whole-square solve kernel, also when the
    right-hand sides need a second, solve-only pass."""
    bl = lib()
    rng = np.random.default_rng(29)
    routes = {sp: cap for sp, cap, _ in bl.routes("f32")}
    for sp, n in routes.items():
        if ":v2=1" not in sp:
            continue
        base = sp.replace(":la=1", "").replace(":v2=1", "")
        A = synth.spd_bbt(rng, n, 777, "f32")
        A[5, n // 3, n // 3] = -1.0
        for nrhs in (3, 11):
            B = synth.rhs_uniform(rng, n, nrhs, 777, "f32")
            for uplo in "LU":
                abuf, a0, bbuf, b0, i0 = call_posv(A, B, uplo, "f32", route=base)
                _, a1, _, b1, i1 = call_posv(A, B, uplo, "f32", route=sp)
                _, x, rinfo = oracle.run(uplo, n, 777, abuf, n, n * n, nrhs, bbuf, n, n * nrhs, threads=THREADS)
                assert np.array_equal(i1, rinfo) and np.array_equal(i0, i1)
                ok = i1 == 0
                X1 = synth.from_colmajor(b1, n, nrhs, 777)
                assert solution_errors(X1[ok], x[ok]).max() <= TOL_X["f32"], sp
                assert np.array_equal(b0.view(np.uint8), b1.view(np.uint8)), (sp, nrhs, uplo)
                f0, f1 = synth.from_colmajor(a0, n, n, 777), synth.from_colmajor(a1, n, n, 777)
                assert np.array_equal(np.ascontiguousarray(f0[ok]).view(np.uint8),
                                      np.ascontiguousarray(f1[ok]).view(np.uint8)), (sp, nrhs, uplo)
