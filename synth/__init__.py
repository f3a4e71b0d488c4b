"""Seeded synthetic inputs for batched Cholesky (potrf) and the SPD solve (posv).

This module is shared by the CPU oracle tests and the CUDA path's tests and benchmark.
It builds Hermitian positive-definite batches and right-hand sides and lays them out
column-major; it contains none of the factorisation or solve arithmetic.

Construction recipes (BatchLAS "Batched Cholesky (potrf)" page, which measures seeded
synthetic SPD batches over grids of n and batch; the concrete recipes below are the ones
this library's workloads name):

* ``bbt``:  A = B*B^H + n*I, B real entries i.i.d. uniform[-1, 1]  (real dtypes), or
  B real and imaginary parts i.i.d. N(0, 1) (complex dtypes).
* ``haar``: A = Q*diag(lam)*Q^T, Q Haar-random orthogonal (QR of an N(0,1) matrix with the
  sign correction Q <- Q*diag(sign(diag R))), lam = 10**(3*U[0,1)), so 1 <= lam < 1e3.

Every matrix is built in float64/complex128, symmetrised as (A + A^H)/2 with a real
diagonal, then rounded to the target dtype, so the stored matrix is exactly Hermitian and the
Lower and Upper triangles describe the same matrix.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

DTYPES = {
    "f32": np.float32,
    "f64": np.float64,
    "c64": np.complex64,
    "c128": np.complex128,
}
WIDE = {"f32": np.float64, "f64": np.float64, "c64": np.complex128, "c128": np.complex128}


def is_complex(dtype: str) -> bool:
    return dtype in ("c64", "c128")


def _hermitian_round(a: np.ndarray, dtype: str) -> np.ndarray:
    """(A + A^H)/2 with a real diagonal, rounded to ``dtype``. a: (batch, n, n) wide."""
    a = 0.5 * (a + np.conj(np.swapaxes(a, -1, -2)))
    if is_complex(dtype):
        idx = np.arange(a.shape[-1])
        a[..., idx, idx] = a[..., idx, idx].real
    return a.astype(DTYPES[dtype])


def spd_bbt(rng: np.random.Generator, n: int, batch: int, dtype: str) -> np.ndarray:
    """A = B*B^H + n*I per item; returns logical matrices (batch, n, n) in ``dtype``."""
    if is_complex(dtype):
        b = rng.standard_normal((batch, n, n)) + 1j * rng.standard_normal((batch, n, n))
    else:
        b = rng.uniform(-1.0, 1.0, (batch, n, n))
    a = b @ np.conj(np.swapaxes(b, -1, -2))
    a = a + n * np.eye(n)
    return _hermitian_round(a, dtype)


def spd_haar(rng: np.random.Generator, n: int, batch: int, dtype: str,
             log10_kappa: float = 3.0) -> np.ndarray:
    """A = Q*diag(lam)*Q^T with Haar Q and lam log-uniform in [1, 10**log10_kappa)."""
    g = rng.standard_normal((batch, n, n))
    q, r = np.linalg.qr(g)
    d = np.sign(np.diagonal(r, axis1=-2, axis2=-1))
    d[d == 0] = 1.0
    q = q * d[:, None, :]
    lam = 10.0 ** (log10_kappa * rng.uniform(0.0, 1.0, (batch, n)))
    a = (q * lam[:, None, :]) @ np.swapaxes(q, -1, -2)
    if is_complex(dtype):
        a = a.astype(np.complex128)
    return _hermitian_round(a, dtype)


def rhs_uniform(rng: np.random.Generator, n: int, nrhs: int, batch: int, dtype: str) -> np.ndarray:
    """Right-hand sides (batch, n, nrhs): entries (and for complex, both parts) uniform[-1,1]."""
    if is_complex(dtype):
        b = rng.uniform(-1.0, 1.0, (batch, n, nrhs)) + 1j * rng.uniform(-1.0, 1.0, (batch, n, nrhs))
    else:
        b = rng.uniform(-1.0, 1.0, (batch, n, nrhs))
    return b.astype(DTYPES[dtype])


# ----------------------------------------------------------------------------- layout

def to_colmajor(a: np.ndarray, ld: Optional[int] = None, stride: Optional[int] = None,
                fill=0) -> np.ndarray:
    """Lay out logical matrices a[b, i, j] (batch, m, k) column-major in a flat buffer:
    element (i, j) of item b at ``b*stride + j*ld + i``. Gaps are set to ``fill``."""
    batch, m, k = a.shape
    ld = m if ld is None else ld
    stride = ld * k if stride is None else stride
    if ld < m or stride < ld * k:
        raise ValueError("ld/stride too small")
    buf = np.full(stride * batch, fill, dtype=a.dtype) if batch else np.zeros(0, a.dtype)
    if batch:
        view = np.lib.stride_tricks.as_strided(
            buf, shape=(batch, k, m),
            strides=(stride * buf.itemsize, ld * buf.itemsize, buf.itemsize))
        view[...] = np.swapaxes(a, -1, -2)
    return buf


def from_colmajor(buf: np.ndarray, m: int, k: int, batch: int, ld: Optional[int] = None,
                  stride: Optional[int] = None) -> np.ndarray:
    """Inverse of :func:`to_colmajor`: returns logical (batch, m, k) copies."""
    ld = m if ld is None else ld
    stride = ld * k if stride is None else stride
    view = np.lib.stride_tricks.as_strided(
        buf, shape=(batch, k, m),
        strides=(stride * buf.itemsize, ld * buf.itemsize, buf.itemsize))
    return np.ascontiguousarray(np.swapaxes(view, -1, -2))


# ----------------------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    """One named synthetic workload: the logical inputs plus the planted expectations."""
    name: str
    dtype: str
    n: int
    batch: int
    uplos: tuple
    A: np.ndarray                     # (batch, n, n) logical, dtype
    nrhs: int = 0
    B: Optional[np.ndarray] = None    # (batch, n, nrhs) logical, dtype
    planted_info: Optional[np.ndarray] = None   # int32 (batch,), 0 where nothing planted


def _planted(a: np.ndarray, first: int, count: int) -> np.ndarray:
    """Items first+k (k < count) get A(k,k) = -1; returns the expected info vector."""
    info = np.zeros(a.shape[0], np.int32)
    for k in range(count):
        a[first + k, k, k] = -1
        info[first + k] = k + 1
    return info


def workload(name: str, batch: Optional[int] = None) -> Workload:
    """Build a named workload. ``batch`` overrides the item count (a leading sub-batch of the
    same seeded stream is NOT implied: a different batch draws a different stream)."""
    specs = {
        # potrf f32 Lower n=8, batch 1024, plus 8 items with A(k,k) = -1 (expected info k+1)
        "f32_n8": dict(dtype="f32", n=8, batch=1024, seed=0, kind="bbt", uplos=("L",), planted=8),
        # potrf f32 n=32 batch 16384, Lower and Upper; posv nrhs=4
        "f32_n32": dict(dtype="f32", n=32, batch=16384, seed=1, kind="bbt", uplos=("L", "U"), nrhs=4),
        # potrf f64 Lower at the +1 rungs, Haar Q, kappa <= 1e3
        "f64_n17": dict(dtype="f64", n=17, batch=32768, seed=2, kind="haar", uplos=("L",)),
        "f64_n33": dict(dtype="f64", n=33, batch=16384, seed=2, kind="haar", uplos=("L",)),
        "f64_n65": dict(dtype="f64", n=65, batch=8192, seed=2, kind="haar", uplos=("L",)),
        # potrf c64 Lower n=128 batch 8192; posv nrhs=8
        "c64_n128": dict(dtype="c64", n=128, batch=8192, seed=3, kind="bbt", uplos=("L",), nrhs=8),
        # potrf f32 / f64 Lower n=512 batch 1024; posv f64 nrhs=8
        "f32_n512": dict(dtype="f32", n=512, batch=1024, seed=4, kind="bbt", uplos=("L",)),
        "f64_n512": dict(dtype="f64", n=512, batch=1024, seed=4, kind="bbt", uplos=("L",), nrhs=8),
    }
    if name not in specs:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(specs)}")
    s = specs[name]
    nb = s["batch"] if batch is None else batch
    rng = np.random.default_rng(s["seed"])
    planted = s.get("planted", 0)
    total = nb + planted
    gen = spd_bbt if s["kind"] == "bbt" else spd_haar
    a = gen(rng, s["n"], total, s["dtype"])
    info = _planted(a, nb, planted) if planted else None
    nrhs = s.get("nrhs", 0)
    b = rhs_uniform(rng, s["n"], nrhs, total, s["dtype"]) if nrhs else None
    return Workload(name=name, dtype=s["dtype"], n=s["n"], batch=total, uplos=s["uplos"],
                    A=a, nrhs=nrhs, B=b, planted_info=info)


WORKLOADS = ("f32_n8", "f32_n32", "f64_n17", "f64_n33", "f64_n65", "c64_n128",
             "f32_n512", "f64_n512")
