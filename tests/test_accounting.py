"""Byte and flop accounting of the benchmark line and the per-workload report, pinned to the
per-configuration figures worked out independently in the measurement specification (bytes of
the referenced triangle at 32-byte sectors, read and written, plus the 4-byte info; LAPACK flop
counts; posv adds B read and written and two triangular solves per right-hand side), and the
report's choice of the binding roof. Runs without a GPU."""
import types

import pytest

import bench
from matrix_dense_linear_spd_gb300 import report

# (dtype, n, nrhs) -> (full storage bytes 2 n^2 s + 4, triangle-sector bytes, flops) per matrix
SPEC = {
    ("f32", 8, 0): (516, 516, 204),
    ("f32", 32, 0): (8196, 5124, 11440),
    ("f32", 32, 4): (9220, 6148, 19504),
    ("f64", 17, 0): (4628, 3140, 1785),
    ("f64", 33, 0): (17428, 10308, 12529),
    ("f64", 65, 0): (67604, 36932, 93665),
    ("c64", 128, 0): (262148, 135172, 2845568),
    ("c64", 128, 8): (278532, 151556, 3892096),
    ("f32", 512, 0): (2097156, 1064964, 44870400),
    ("f64", 512, 0): (4194308, 2113540, 44870400),
    ("f64", 512, 8): (4259844, 2179076, 49060608),
}
ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}


@pytest.mark.parametrize("key", sorted(SPEC), ids=lambda k: f"{k[0]}_n{k[1]}_nrhs{k[2]}")
def test_bytes_and_flops_match_the_specification(key):
    dtype, n, nrhs = key
    full, tri, fl = SPEC[key]
    rhs = 2 * n * nrhs * ESIZE[dtype]
    assert 2 * n * n * ESIZE[dtype] + 4 + rhs == full
    assert 2 * report.tri_sector_bytes(n, dtype, "L") + 4 + rhs == tri
    assert report.flops(n, dtype, nrhs) == pytest.approx(fl, abs=0.5)
    if nrhs == 0:
        assert bench.potrf_bytes(n, dtype) == tri
        assert bench.potrf_flops(n, dtype) == pytest.approx(fl, abs=0.5)


def test_triangle_bytes_agree_between_modules_and_are_bounded():
    # Lower touches rows c..n-1 of column c, Upper rows 0..c: different sectors of a column-major
    # item. Both modules count each triangle's own sectors alike, and the count lies between the
    # packed triangle and the full square.
    for n, dt in ((32, "f32"), (8, "f32"), (17, "f64")):
        lo, up = bench.triangle_sector_bytes(n, dt, "L"), bench.triangle_sector_bytes(n, dt, "U")
        assert lo == report.tri_sector_bytes(n, dt, "L") and up == report.tri_sector_bytes(n, dt, "U")
        assert n * (n + 1) // 2 * ESIZE[dt] <= min(lo, up) <= n * n * ESIZE[dt]


def _row(dtype, n, batch, ms, route, nrhs=0):
    w = types.SimpleNamespace(n=n, batch=batch, dtype=dtype)
    m = {"ms": ms, "rel_sd": 0.01, "iso": ms, "vms": None, "route": route, "info_ok": True, "l2_resident": False}
    cells = [c.strip() for c in report.row("w", w, "potrf" if not nrhs else "posv", "L", nrhs, m,
                                           6786.9, 80.4, 405.7, 1.26).split("|")[1:-1]]
    return cells[9], float(cells[10])          # binding roof, roof fraction


def test_binding_roof_and_fraction():
    # f32 n=32 b16384 in 23.0 us: HBM binds (5,124 B at 6,787 GB/s is far above 11,440 flops at
    # 80.4 TF/s); fraction = 5124 * 16384 / 6786.9e9 / 23.0e-6
    bind, frac = _row("f32", 32, 16384, 0.0230, "warp:p=16:r=2:full=1:x2=1:la=1:v2=1")
    assert bind == "HBM" and frac == pytest.approx(5124 * 16384 / 6786.9e9 / 23.0e-6, abs=0.006)
    # f64 n=512 b1024 in 47.2 ms: FP64 binds; fraction = 44,870,400 * 1024 / 1.26e12 / 47.2e-3
    bind, frac = _row("f64", 512, 1024, 47.2, "blocked:nb=32")
    assert bind == "FP64" and frac == pytest.approx(44870400 * 1024 / 1.26e12 / 47.2e-3, abs=0.006)
    # the tensor-core route takes the 3xTF32 rate: at f32 n=512 HBM then binds
    bind, _ = _row("f32", 512, 1024, 1.45, "blocked:nb=32:tc=2")
    assert bind == "HBM"
    # the SIMT route at the same shape is bound by FP32
    bind, _ = _row("f32", 512, 1024, 5.2, "blocked:nb=32")
    assert bind == "FP32"
