"""Host-side tests of the tuner's ledger -> table step (BatchLAS "Flat kernel selection",
section 6.4, table regeneration) and of its edge refinement along n: no GPU. A synthetic
ledger goes through ledger_to_tables / format_table, the ranking, ties, re-measurement and
header are checked, and the written table is read back by the library's own selection layer."""
import json
import os
import subprocess
import sys

import pytest

from matrix_dense_linear_spd_gb300 import sweep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def rec(cand, ms, n=32, batch=16384, uplo="L", dtype="f32", attempt=0, run=1.0, op="potrf", nrhs=0, kind="time"):
    return {"op": op, "device": "sm_999", "dtype": dtype, "uplo": uplo, "n": n, "nrhs": nrhs, "batch": batch,
            "candidate": cand, "ms": ms, "attempt": attempt, "run": run, "kind": kind}


def test_ranking_is_by_median_and_ties_by_spelling():
    recs = [rec("warp:p=8:r=4", 0.03), rec("warp:p=8:r=4", 0.02), rec("warp:p=8:r=4", 0.05),   # median 0.03
            rec("tile:p=4:s=8", 0.04), rec("tile:p=4:s=8", 0.01), rec("tile:p=4:s=8", 0.02),   # median 0.02
            rec("blocked:nb=32", 0.03), rec("blocked:nb=32", 0.03),                           # median 0.03: tie
            rec("tile:p=2:s=4", 9.0, kind="rejected")]
    rows = sweep.ledger_to_tables(recs)["potrf"]
    assert len(rows) == 1
    key, ranked = rows[0]
    assert key == {"dtype": "f32", "uplo": "L", "n": 32, "batch": 16384}
    assert [sp for sp, _ in ranked] == ["tile:p=4:s=8", "blocked:nb=32", "warp:p=8:r=4"]
    assert ranked[0][1] == pytest.approx(0.02)


def test_latest_measurement_of_a_cell_replaces_earlier_ones():
    recs = [rec("a:x=1", 1.0, attempt=0), rec("b:x=1", 2.0, attempt=0),
            rec("a:x=1", 3.0, attempt=1), rec("b:x=1", 2.5, attempt=1),        # re-measured: b wins
            rec("a:x=1", 0.5, run=0.5, attempt=3)]                             # an older run: ignored
    (_, ranked), = sweep.ledger_to_tables(recs)["potrf"]
    assert [sp for sp, _ in ranked] == ["b:x=1", "a:x=1"]
    assert ranked[0][1] == 2.5


def test_rows_are_ordered_and_posv_rows_carry_nrhs():
    recs = [rec("x", 1.0, n=64, dtype="f64"), rec("x", 1.0, n=8), rec("x", 1.0, n=32, uplo="U"),
            rec("y", 1.0, n=16, op="posv", nrhs=4), rec("y", 1.0, n=16, op="posv", nrhs=1)]
    t = sweep.ledger_to_tables(recs)
    assert [(k["dtype"], k["uplo"], k["n"]) for k, _ in t["potrf"]] == [("f32", "L", 8), ("f32", "U", 32), ("f64", "L", 64)]
    assert [k["nrhs"] for k, _ in t["posv"]] == [1, 4]
    text = sweep.format_table("posv", "sm_999", t["posv"], "posv.sm_999.jsonl", date="2026-01-01")
    lines = text.splitlines()
    assert lines[0].startswith("# op=posv device=sm_999 source=ledger:posv.sm_999.jsonl date=2026-01-01")
    assert lines[1] == "# keys: dtype:exact uplo:exact n:log:3 nrhs:log batch:log"
    assert lines[2] == "dtype=f32 uplo=L n=16 nrhs=1 batch=16384 | y 1.00000 # measured"


def test_edge_refinement_midpoints():
    w = [(4, "a"), (8, "a"), (16, "b"), (17, "c"), (32, "c"), (64, "d")]
    assert sweep.bisect_points(w) == [12, 48]          # 16 -> 17 is adjacent: nothing to refine


def test_written_table_drives_the_selection_layer(tmp_path):
    """A ledger whose winner at f32 n=32 is tile:p=4:s=8 (slower elsewhere) yields a table that the
    library reads (BL_TUNED_DIR) and follows, in a fresh process (the table cache is per process)."""
    recs = [rec("tile:p=4:s=8", 0.010), rec("warp:p=16:r=2", 0.020),
            rec("warp:p=16:r=2", 0.010, n=8), rec("tile:p=4:s=8", 0.030, n=8)]
    ledger = tmp_path / "potrf.sm_999.jsonl"
    ledger.write_text("\n".join(json.dumps(r) for r in recs) + "\n")
    paths = sweep.write_tables(str(ledger), str(tmp_path))
    assert paths == [str(tmp_path / "potrf.sm_999.txt")]
    code = r"""
import matrix_dense_linear_spd_gb300 as bl
print(bl.select_debug("potrf", "f32", "L", 32, 0, 16384, devkey="sm_999"))
print(bl.select_debug("potrf", "f32", "L", 8, 0, 16384, devkey="sm_999"))
"""
    env = dict(os.environ, BL_TUNED_DIR=str(tmp_path), PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    a, b = out.stdout.strip().splitlines()
    assert a.startswith("tile:p=4:s=8 [table override sm_999 row n=32 batch=16384]")
    assert b.startswith("warp:p=16:r=2 [table override sm_999 row n=8 batch=16384]")


def test_shipped_tables_are_the_verdict_of_the_committed_ledgers(tmp_path):
    """Every shipped table row is what the ledger -> table step makes of the committed ledgers
    (tuned/ledger, all runs, the latest measurement of a cell and candidate winning): the tables
    are reproducible from the measurements alone (only the header's date may differ)."""
    import re
    tuned = os.path.join(os.path.dirname(sweep.__file__), "tuned")
    for op in ("potrf", "posv"):
        ledgers = sweep.shipped_ledgers(op)
        assert ledgers, op
        (path,) = sweep.write_tables(",".join(ledgers), str(tmp_path))
        got = open(path).read()
        shipped = open(os.path.join(tuned, f"{op}.sm_103.txt")).read()
        assert re.sub(r"date=\S+", "", got) == re.sub(r"date=\S+", "", shipped), op


# (op, dtype, uplo, n, nrhs, batch) of every configuration the benchmark and the report time
CONFIG_CELLS = [
    ("potrf", "f32", "L", 8, 0, 1024), ("potrf", "f32", "L", 32, 0, 16384), ("potrf", "f32", "U", 32, 0, 16384),
    ("posv", "f32", "L", 32, 4, 16384), ("potrf", "f64", "L", 17, 0, 32768), ("potrf", "f64", "L", 33, 0, 16384),
    ("potrf", "f64", "L", 65, 0, 8192), ("potrf", "c64", "L", 128, 0, 8192), ("posv", "c64", "L", 128, 8, 8192),
    ("potrf", "f32", "L", 512, 0, 1024), ("potrf", "f64", "L", 512, 0, 1024), ("posv", "f64", "L", 512, 8, 1024),
]


def test_every_configuration_is_a_measured_row_and_selects_its_winner():
    """Each configuration's own (dtype, uplo, n[, nrhs], batch) is a measured row of the shipped
    table (not a nearest-row borrow), and the selection layer picks that row's winner there."""
    import matrix_dense_linear_spd_gb300 as bl
    tuned = os.path.join(os.path.dirname(sweep.__file__), "tuned")
    rows = {}
    for op in ("potrf", "posv"):
        for line in open(os.path.join(tuned, f"{op}.sm_103.txt")):
            if line.startswith("#"):
                continue
            key, rest = line.split("|", 1)
            rows[(op, key.strip())] = rest.split("|")[0].strip().rsplit(" ", 1)[0]
    for op, dt, uplo, n, nrhs, batch in CONFIG_CELLS:
        key = f"dtype={dt} uplo={uplo} n={n}" + (f" nrhs={nrhs}" if op == "posv" else "") + f" batch={batch}"
        assert (op, key) in rows, (op, key)
        chosen = bl.select_debug(op, dt, uplo, n, nrhs, batch)
        assert chosen.split(" ")[0] == rows[(op, key)], (op, key, chosen)
