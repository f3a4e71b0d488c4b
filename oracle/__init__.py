"""CPU oracle for batched potrf / posv / potrs (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package. It wraps ``bl_oracle.c`` -- a plain long-double Cholesky-Banachiewicz plus
forward/back substitution written from the BatchLAS "Batched Cholesky (potrf)" page -- and
shares no code with the CUDA library.

Parity status: every function here is pinned by ``tests/test_oracle.py`` (integer-exact
factor recovery, closed forms, planted failures, brute-force leading minors, a LAPACK third
opinion and residual invariants). Nothing is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bl_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile bl_oracle.c into liboracle.so with gcc (plain C, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.bl_oracle_run.restype = ctypes.c_int
            lib.bl_oracle_run.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.bl_oracle_ldbl_mant_dig.restype = ctypes.c_int
            _lib = lib
    return _lib


def long_double_digits() -> int:
    """Mantissa bits of the oracle's long double (64: x87 extended; 113: binary128)."""
    return _load().bl_oracle_ldbl_mant_dig()


def _is_complex(arr: np.ndarray) -> bool:
    return np.iscomplexobj(arr)


def _as_double_buffer(buf: np.ndarray) -> np.ndarray:
    """Promote a flat column-major buffer of f32/f64/c64/c128 values to double storage
    (complex: interleaved re/im). Promotion is exact."""
    if _is_complex(buf):
        return np.ascontiguousarray(buf.astype(np.complex128)).view(np.float64)
    return np.ascontiguousarray(buf.astype(np.float64))


def run(uplo: str, n: int, batch: int, a_buf: np.ndarray, lda: int, stride_a: int,
        nrhs: int = 0, b_buf: np.ndarray | None = None, ldb: int = 0, stride_b: int = 0,
        factor_given: bool = False, want_factor: bool = True, threads: int = 1):
    """Run the oracle on column-major buffers laid out exactly as the library receives them.

    Returns (factor, x, info):
      factor -- (batch, n, n) long double / clongdouble logical matrices holding the factor in
                the referenced triangle (zeros elsewhere), or None;
      x      -- (batch, n, nrhs) solutions (right-hand sides unchanged where info > 0), or None;
      info   -- int32 (batch,).
    """
    if uplo not in ("L", "U"):
        raise ValueError("uplo must be 'L' or 'U'")
    cplx = _is_complex(a_buf)
    lib = _load()
    a_d = _as_double_buffer(a_buf)
    b_d = _as_double_buffer(b_buf) if (nrhs and b_buf is not None) else None
    sc = 2 if cplx else 1
    out_f = np.zeros(batch * n * n * sc, np.longdouble) if want_factor else None
    out_x = np.zeros(batch * n * nrhs * sc, np.longdouble) if nrhs else None
    info = np.zeros(batch, np.int32)
    rc = lib.bl_oracle_run(
        int(cplx), int(uplo == "U"), int(factor_given), n, batch,
        a_d.ctypes.data, lda, stride_a, nrhs,
        b_d.ctypes.data if b_d is not None else None, ldb, stride_b,
        out_f.ctypes.data if out_f is not None else None,
        out_x.ctypes.data if out_x is not None else None,
        info.ctypes.data, max(1, int(threads)))
    if rc != 0:
        raise MemoryError("oracle worker failed to allocate scratch")

    def logical(flat, rows, cols):
        if flat is None:
            return None
        if cplx:
            c = np.empty(flat.size // 2, np.clongdouble)
            c.real = flat[0::2]
            c.imag = flat[1::2]
            flat = c
        return np.swapaxes(flat.reshape(batch, cols, rows), -1, -2)

    return logical(out_f, n, n), logical(out_x, n, nrhs) if nrhs else None, info


def potrf(A: np.ndarray, uplo: str = "L", threads: int = 1):
    """Factor logical matrices A (batch, n, n) (any of the four dtypes). Only the referenced
    triangle of A is read. Returns (factor, info)."""
    from synth import to_colmajor
    batch, n, _ = A.shape
    f, _, info = run(uplo, n, batch, to_colmajor(A), n, n * n, threads=threads)
    return f, info


def posv(A: np.ndarray, B: np.ndarray, uplo: str = "L", threads: int = 1):
    """Factor and solve A X = B for logical A (batch, n, n), B (batch, n, nrhs).
    Returns (factor, X, info)."""
    from synth import to_colmajor
    batch, n, _ = A.shape
    nrhs = B.shape[-1]
    return run(uplo, n, batch, to_colmajor(A), n, n * n, nrhs, to_colmajor(B), n, n * nrhs,
               threads=threads)


def potrs(F: np.ndarray, B: np.ndarray, uplo: str = "L", threads: int = 1):
    """Solve with a given factor F (batch, n, n) held in its referenced triangle.
    Returns X (batch, n, nrhs)."""
    from synth import to_colmajor
    batch, n, _ = F.shape
    nrhs = B.shape[-1]
    _, x, _ = run(uplo, n, batch, to_colmajor(F), n, n * n, nrhs, to_colmajor(B), n, n * nrhs,
                  factor_given=True, want_factor=False, threads=threads)
    return x
