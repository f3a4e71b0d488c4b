"""Armed breaks for the oracle's pins: plant one plausible mistake at a time in a copy of the
oracle's C source, build it, and check that the pin battery goes red. A pin set that stays
green under a planted defect could not have caught it (BatchLAS "Batched Cholesky (potrf)"
page, "Armed breaks (R9)": every guard is planted, observed red and restored).

The mutants live only in a temporary directory; the committed oracle is never modified.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "bl_oracle.c")

# (name, exact text in bl_oracle.c, replacement)
MUTANTS = [
    ("drop_conj_offdiag", "s -= l[k * n + i] * conjl(l[k * n + j]);", "s -= l[k * n + i] * l[k * n + j];"),
    ("info_zero_based", "if (!(d > 0)) return i + 1;\n        l[i * n + i] = sqrtl(d);\n    }\n    return 0;\n}\n\nstatic int64_t chol_cplx",
     "if (!(d > 0)) return i;\n        l[i * n + i] = sqrtl(d);\n    }\n    return 0;\n}\n\nstatic int64_t chol_cplx"),
    ("wrong_sign_pivot", "d -= l[k * n + i] * l[k * n + i];", "d += l[k * n + i] * l[k * n + i];"),
    ("dropped_first_term", "for (int64_t k = 0; k < j; ++k) s -= l[k * n + i] * l[k * n + j];",
     "for (int64_t k = 1; k < j; ++k) s -= l[k * n + i] * l[k * n + j];"),
    ("upper_reads_lower", "return upper ? (ldr)a[i * ld + c] : (ldr)a[c * ld + i];",
     "return (ldr)a[c * ld + i];"),
    ("nan_pivot_passes", "if (!(d > 0)) return i + 1;\n        l[i * n + i] = sqrtl(d);\n    }\n    return 0;\n}\n\nstatic int64_t chol_cplx",
     "if (d <= 0) return i + 1;\n        l[i * n + i] = sqrtl(d);\n    }\n    return 0;\n}\n\nstatic int64_t chol_cplx"),
    ("back_solve_no_conj", "s -= conjl(l[i * n + k]) * x[k];", "s -= l[i * n + k] * x[k];"),
    ("forward_transposed", "for (int64_t k = 0; k < i; ++k) s -= l[k * n + i] * x[k];\n        x[i] = s / l[i * n + i];",
     "for (int64_t k = 0; k < i; ++k) s -= l[i * n + k] * x[k];\n        x[i] = s / l[i * n + i];"),
    ("upper_store_no_conj", "if (upper) v = conjl(v);", ""),
    ("failed_solve_not_skipped", "if (!info) solve_real(n, l, x);", "solve_real(n, l, x);"),
]


def _battery():
    """The pins that each mutant must trip (any one failing is enough)."""
    yield lambda: [pins.test_integer_factor_is_recovered_exactly(dt, u, n)
                   for dt in ("f64", "c128") for u in "LU" for n in (3, 7)]
    yield lambda: pins.test_info_matches_brute_force_leading_minors()
    yield lambda: [pins.test_planted_failures(dt) for dt in ("f64", "c128")]
    yield lambda: [pins.test_posv_integer_solution_is_exact(c, u) for c in (False, True) for u in "LU"]
    yield lambda: pins.test_posv_closed_forms_and_failure()
    yield lambda: [pins.test_lapack_third_opinion(dt, "bbt", u) for dt in ("f64", "c128") for u in "LU"]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text not unique/absent"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(path), "-lm", "-lpthread"], check=True)
    lib = ctypes.CDLL(str(so))
    ref = oracle._load()
    lib.bl_oracle_run.restype = ref.bl_oracle_run.restype
    lib.bl_oracle_run.argtypes = ref.bl_oracle_run.argtypes
    lib.bl_oracle_ldbl_mant_dig.restype = ctypes.c_int
    return lib


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_every_planted_oracle_defect_is_caught(tmp_path, monkeypatch, name, old, new):
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = 0
    for check in _battery():
        try:
            check()
        except (AssertionError, np.linalg.LinAlgError):
            caught += 1
    assert caught >= 1, f"planted defect {name!r} left every pin green"


def test_unmutated_battery_is_green():
    for check in _battery():
        check()
