"""Host-side tests of the C ABI (no GPU): the library loads and exports every symbol the
header declares, argument errors are caught on the host before any CUDA call, and the flat
selection layer (BatchLAS "Flat kernel selection": tables, nearest row, can_run, pins) picks as
specified for a synthetic device.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bl.h")


@pytest.fixture(scope="module")
def bl():
    import matrix_dense_linear_spd_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from matrix_dense_linear_spd_gb300 import build
        build.build()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bl_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(bl):
    names = declared_functions()
    assert {"bl_potrf", "bl_posv", "bl_potrs", "bl_status_string"} <= set(names)
    lib = ctypes.CDLL(bl.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in bl.h but not exported"
    assert set(bl.EXPORTED) >= set(names)


def test_status_strings_and_version(bl):
    lib = bl.get_lib()
    for code in range(5):
        assert lib.bl_status_string(code)
    assert lib.bl_status_string(99) == b"unknown status"
    assert lib.bl_version() >= 100


INVALID = [
    # (op, dtype, uplo, n, nrhs, batch)
    ("potrf", "f32", "L", 0, 0, 1),
    ("potrf", "f32", "L", -3, 0, 1),
    ("potrf", "f32", "L", 4, 0, 0),
    ("potrf", "f64", "U", (1 << 20) + 1, 0, 1),
    ("posv", "c64", "L", 4, 0, 1),
    ("potrs", "c128", "U", 4, -1, 1),
]


@pytest.mark.parametrize("case", INVALID)
def test_invalid_sizes_are_rejected_on_the_host(bl, case):
    op, dt, uplo, n, nrhs, batch = case
    out = bl.select_debug(op, dt, uplo, n, nrhs, batch)
    assert out.startswith("error:"), out


def test_invalid_pointers_strides_and_enums_are_rejected_without_a_gpu(bl):
    lib = bl.get_lib()
    fake = 256  # never dereferenced: validation fails first
    assert lib.bl_potrf(0, 0, 4, 1, None, 4, 16, fake, None) == 1
    assert lib.bl_potrf(0, 0, 4, 1, fake, 3, 16, fake, None) == 1           # lda < n
    assert lib.bl_potrf(0, 0, 4, 2, fake, 4, 15, fake, None) == 1           # items overlap
    assert lib.bl_potrf(0, 0, 4, 1, fake, 4, 16, None, None) == 1           # info NULL
    assert lib.bl_potrf(2, 0, 4, 1, fake, 4, 16, fake, None) == 1           # uplo
    assert lib.bl_potrf(0, 7, 4, 1, fake, 4, 16, fake, None) == 1           # dtype
    assert lib.bl_posv(0, 0, 4, 2, 1, fake, 4, 16, None, 4, 8, fake, None) == 1  # B NULL
    assert lib.bl_posv(0, 0, 4, 2, 1, fake, 4, 16, fake, 3, 8, fake, None) == 1  # ldb < n
    assert lib.bl_posv(0, 0, 4, 2, 2, fake, 4, 16, fake, 4, 7, fake, None) == 1  # B items overlap
    assert lib.bl_potrs(0, 0, 4, 0, 1, fake, 4, 16, fake, 4, 4, None) == 1      # nrhs 0
    assert lib.bl_potrf(0, 1, 4, 1, fake + 4, 4, 16, fake, None) == 1       # f64 A not 8-aligned
    assert lib.bl_potrf(0, 3, 4, 1, fake + 8, 4, 16, fake, None) == 1       # c128 A not 16-aligned
    assert lib.bl_potrf(0, 0, 4, 1, fake, 4, 16, fake + 2, None) == 1       # info not 4-aligned
    assert lib.bl_posv(0, 1, 4, 2, 1, fake, 4, 16, fake + 4, 4, 8, fake, None) == 1  # B not 8-aligned
    assert b"lda" in lib.bl_last_error() or lib.bl_last_error()
    assert lib.bl_set_route(b"getrf", b"tile:p=4:s=8") == 1


def test_can_run_is_capacity_only(bl):
    """A tile variant holds n + (right-hand sides per pass) <= P*S; blocked holds any n."""
    for dt in ("f32", "f64", "c64", "c128"):
        routes = bl.routes(dt)
        assert any(cap == 0 for _, cap, _ in routes), "a blocked variant must exist"
        for sp, cap, rhs in routes:
            bl.set_route("potrf", sp)
            try:
                if cap:
                    assert bl.select_debug("potrf", dt, "L", cap, 0, 7).startswith(sp + " [pin]")
                    assert bl.select_debug("potrf", dt, "U", cap + 1, 0, 7).startswith("error:")
                else:
                    assert bl.select_debug("potrf", dt, "U", 1000, 0, 7).startswith(sp + " [pin]")
            finally:
                bl.set_route("potrf", None)
            if cap and rhs < 0:                  # factor-only variant: a solve pin is refused
                bl.set_route("posv", sp)
                try:
                    assert bl.select_debug("posv", dt, "L", 2, 1, 7).startswith("error:")
                finally:
                    bl.set_route("posv", None)
            elif cap and sp.startswith("warp"):   # right-hand sides do not take tile rows
                bl.set_route("posv", sp)
                try:
                    assert bl.select_debug("posv", dt, "L", cap, 50, 7).startswith(sp)
                    assert bl.select_debug("posv", dt, "L", cap + 1, 1, 7).startswith("error:")
                finally:
                    bl.set_route("posv", None)
            elif cap:
                bl.set_route("posv", sp)
                try:
                    assert bl.select_debug("posv", dt, "L", cap - rhs, 50, 7).startswith(sp)
                    assert bl.select_debug("posv", dt, "L", cap - rhs + 1, 50, 7).startswith("error:")
                    assert bl.select_debug("posv", dt, "L", cap - 1, 1, 7).startswith(sp)
                finally:
                    bl.set_route("posv", None)


def test_pins_parse_and_unknown_pins_fail(bl):
    bl.set_route("potrf", " TILE:4:8 ")
    try:
        assert bl.select_debug("potrf", "f32", "L", 30, 0, 100).startswith("tile:p=4:s=8 [pin]")
    finally:
        bl.set_route("potrf", None)
    for bad in ("tile:p=3:s=3", "vendor", "cta", "blocked:nb=7"):
        bl.set_route("potrf", bad)
        try:
            assert bl.select_debug("potrf", "f32", "L", 30, 0, 100).startswith("error:"), bad
        finally:
            bl.set_route("potrf", None)
    bl.set_route("potrf", "auto")
    try:
        assert not bl.select_debug("potrf", "f32", "L", 30, 0, 100).startswith("error:")
    finally:
        bl.set_route("potrf", None)


def test_shared_memory_limit_is_a_can_run_term(bl):
    """A device with little opt-in shared memory cannot run the large variants."""
    out = bl.select_debug("potrf", "c64", "L", 128, 0, 8192, smem_optin=16 * 1024)
    assert out.startswith("error: no kernel can run"), out
    assert bl.select_debug("potrf", "f32", "L", 8, 0, 8192, smem_optin=16 * 1024).startswith(("tile", "warp"))
    assert not bl.select_debug("potrf", "c64", "L", 128, 0, 8192).startswith("error:")


def _write_table(tmp_path, op, text):
    d = tmp_path / "tuned"
    d.mkdir(exist_ok=True)
    (d / f"{op}.sm_999.txt").write_text(text)
    return str(d)


TABLE = """# op=potrf device=sm_999 source=synthetic
# keys: dtype:exact uplo:exact n:log:3 batch:log
dtype=f32 uplo=L n=8 batch=1024 | tile:p=2:s=4 0.01 | tile:p=4:s=4 0.02
dtype=f32 uplo=L n=32 batch=16384 | tile:p=8:s=8 0.03 | tile:p=4:s=8 0.04
dtype=f32 uplo=L n=32 batch=128 | tile:p=4:s=8 0.01 | tile:p=8:s=8 0.02
dtype=f32 uplo=L n=512 batch=1024 | blocked:nb=64 1.0 | blocked:nb=32 1.2
dtype=f32 uplo=U n=32 batch=16384 | tile:p=4:s=9 0.05
dtype=f64 uplo=L n=64 batch=1000 | tile:p=8:s=8 0.1
"""


def test_table_nearest_row_rules(bl, tmp_path, monkeypatch):
    """Run in a subprocess: the table cache and BL_TUNED_DIR are per process."""
    import subprocess
    import sys
    d = _write_table(tmp_path, "potrf", TABLE)
    code = r"""
import matrix_dense_linear_spd_gb300 as bl
q = lambda *a, **k: bl.select_debug(*a, devkey="sm_999", **k)
print(q("potrf", "f32", "L", 32, 0, 16384))
print(q("potrf", "f32", "L", 30, 0, 200))
print(q("potrf", "f32", "L", 9, 0, 1024))
print(q("potrf", "f32", "L", 400, 0, 1024))
print(q("potrf", "f32", "U", 32, 0, 16384))
print(q("potrf", "f32", "U", 33, 0, 16384))
print(q("potrf", "f64", "U", 64, 0, 1000))
print(q("potrf", "c64", "L", 40, 0, 1000))
"""
    env = dict(os.environ, BL_TUNED_DIR=d, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    lines = out.stdout.strip().splitlines()
    assert lines[0].startswith("tile:p=8:s=8 [table override sm_999 row n=32 batch=16384]")
    assert lines[1].startswith("tile:p=4:s=8 [table override sm_999 row n=32 batch=128]")   # batch decides
    assert lines[2].startswith("tile:p=4:s=4")                      # first candidate cannot hold n=9
    assert lines[3].startswith("blocked:nb=64")
    assert lines[4].startswith("tile:p=4:s=9")                      # exact uplo match
    assert lines[5].startswith("tile:p=4:s=9")
    assert lines[6].startswith("tile:p=8:s=8")                      # uplo dropped: nearest f64 row
    assert "last resort" in lines[7]                                # no c64 rows at all


def test_shipped_tables_name_only_compiled_variants(bl):
    tdir = os.path.join(ROOT, "matrix_dense_linear_spd_gb300", "tuned")
    known = {dt: {sp for sp, _, _ in bl.routes(dt)} for dt in ("f32", "f64", "c64", "c128")}
    for f in sorted(os.listdir(tdir)) if os.path.isdir(tdir) else []:
        if not f.endswith(".txt"):
            continue
        keys_seen = False
        for line in open(os.path.join(tdir, f)):
            if line.startswith("# keys:"):
                keys_seen = True
            if not line.strip() or line.startswith("#"):
                continue
            line = line.split("#")[0]
            cells = line.split("|")
            kv = dict(x.split("=") for x in cells[0].split())
            times = []
            for c in cells[1:]:
                parts = c.split()
                assert parts[0] in known[kv["dtype"]], (f, parts[0])
                if len(parts) > 1 and parts[1] != "-":
                    times.append(float(parts[1]))
            assert times == sorted(times) or len(times) < 2 or max(times) / min(times) < 1.5, (f, line)
        assert keys_seen, f


def test_column_block_and_packed_routes_parse_and_select(bl):
    """The column-block tensor-core variant (blocked:nb=32:tc=2, f32 potrf, n <= 512) and the
    packed-FMA lane-row variants (warp:...:x2=1, f32) are compiled, pinnable by their spellings,
    refused where they cannot run, and chosen by the shipped f32 tables where they were fastest."""
    f32 = {sp: (cap, rhs) for sp, cap, rhs in bl.routes("f32")}
    assert f32["blocked:nb=32:tc=2"] == (512, -1)                  # factor only, n <= 512
    for sp in ("warp:p=16:r=2:full=1:x2=1", "warp:p=8:r=4:full=1:x2=1", "warp:p=8:r=2:full=1:x2=1"):
        assert sp in f32, sp
    for other in ("f64", "c64", "c128"):
        assert not any(sp.endswith(":x2=1") or sp.endswith(":tc=2") for sp, _, _ in bl.routes(other))
    for op, sp, n, ok in (("potrf", "blocked:nb=32:tc=2", 512, True), ("potrf", "blocked:nb=32:tc=2", 513, False),
                          ("posv", "blocked:nb=32:tc=2", 64, False), ("potrf", "warp:p=16:r=2:full=1:x2=1", 32, True),
                          ("potrf", "WARP:16:2:1:1", 32, True), ("posv", "warp:p=8:r=4:full=1:x2=1", 28, True)):
        bl.set_route(op, sp)
        try:
            out = bl.select_debug(op, "f32", "L", n, 4 if op == "posv" else 0, 64)
            assert out.startswith("error:") != ok, (op, sp, n, out)
        finally:
            bl.set_route(op, None)
    # the shipped tables route the benchmark shape and the large orders to the new variants
    assert bl.select_debug("potrf", "f32", "L", 32, 0, 16384).startswith("warp:p=16:r=2:full=1:x2=1")
    assert bl.select_debug("potrf", "f32", "L", 512, 0, 1024).startswith("blocked:nb=32:tc=2")
    assert bl.select_debug("potrf", "f32", "U", 512, 0, 1024).startswith("blocked:nb=32:tc=2")
    assert bl.select_debug("posv", "f32", "L", 512, 8, 1024).startswith("blocked:nb=32 ")


def test_thread_variants_parse_and_select(bl):
    """The thread-per-matrix variants -- a lane pair per matrix (thread:n=N:p=2, f64 and c128)
    and fully unrolled at one order (thread:n=N:e=1, f64) -- are compiled, pinnable by their
    spellings (also positionally), refused above their order and for posv (factor only), and
    the shipped f64 table picks the unrolled order-17 variant for the n=17 configuration."""
    f64 = {sp: (cap, rhs) for sp, cap, rhs in bl.routes("f64")}
    c128 = {sp: (cap, rhs) for sp, cap, rhs in bl.routes("c128")}
    assert f64["thread:n=18:p=2"] == (18, -1) and c128["thread:n=18:p=2"] == (18, -1)
    assert f64["thread:n=17:e=1"] == (17, -1)
    assert not any(":e=1" in sp for sp in c128)
    for op, sp, n, ok in (("potrf", "thread:n=17:e=1", 17, True), ("potrf", "thread:n=17:e=1", 18, False),
                          ("potrf", "thread:n=17:e=1", 9, True), ("posv", "thread:n=17:e=1", 17, False),
                          ("potrf", "THREAD:18:2", 18, True), ("potrf", "thread:n=18:p=2", 19, False)):
        bl.set_route(op, sp)
        try:
            out = bl.select_debug(op, "f64", "L", n, 4 if op == "posv" else 0, 4096)
            assert out.startswith("error:") != ok, (op, sp, n, out)
            if ok:
                assert out.startswith("thread:n=17:e=1" if ":e=1" in sp else "thread:n=18:p=2"), out
        finally:
            bl.set_route(op, None)
    assert bl.select_debug("potrf", "f64", "L", 17, 0, 32768).startswith("thread:n=17:e=1")
