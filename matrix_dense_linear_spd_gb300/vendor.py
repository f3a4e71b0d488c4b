"""cuSOLVER's batched Cholesky (``cusolverDn<t>potrfBatched``) through ctypes: the vendor
reference point that the measurement harness times next to this library ("Small-n baseline"
page: the native kernels are compared with the vendor's batched potrf on the same inputs).

It is a reference point only: no route of the library calls it. The routine factors in place
from an array of per-item device pointers, which is built once per buffer, outside any timed
region, exactly as a caller of cuSOLVER would hold it.
"""
from __future__ import annotations

import ctypes
import ctypes.util
import os

_NAMES = ("libcusolver.so.12", "libcusolver.so.11", "libcusolver.so")
_FUNCS = {"f32": "cusolverDnSpotrfBatched", "f64": "cusolverDnDpotrfBatched",
          "c64": "cusolverDnCpotrfBatched", "c128": "cusolverDnZpotrfBatched"}
ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}


def _open():
    errs = []
    cands = list(_NAMES)
    for d in (os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/lib64", "/usr/local/cuda/lib64"):
        cands += [os.path.join(d, nm) for nm in _NAMES]
    try:
        import torch
        tl = os.path.join(os.path.dirname(torch.__file__), "..", "nvidia")
        for sub in ("cu13/lib", "cusolver/lib"):
            cands += [os.path.join(tl, sub, nm) for nm in _NAMES]
    except Exception:
        pass
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError as e:
            errs.append(str(e))
    raise OSError("cuSOLVER not found: " + "; ".join(errs[:3]))


class CusolverPotrfBatched:
    """potrfBatched on a torch device buffer holding `batch` items at a fixed item stride."""

    def __init__(self):
        self.lib = _open()
        self.handle = ctypes.c_void_p()
        st = self.lib.cusolverDnCreate(ctypes.byref(self.handle))
        if st != 0:
            raise RuntimeError(f"cusolverDnCreate failed: {st}")
        for f in _FUNCS.values():
            getattr(self.lib, f).argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            getattr(self.lib, f).restype = ctypes.c_int
        self.lib.cusolverDnSetStream.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        self._arrays = {}

    def pointer_array(self, base: int, batch: int, stride: int, dtype: str, device):
        """Device int64 array of item pointers base + b*stride*esize (built once per buffer)."""
        import torch
        key = (base, batch, stride, dtype)
        if key not in self._arrays:
            offs = torch.arange(batch, dtype=torch.int64, device=device) * (stride * ESIZE[dtype])
            self._arrays[key] = offs + base
        return self._arrays[key]

    def potrf(self, uplo: str, dtype: str, n: int, batch: int, ptrs, lda: int, info_ptr: int, stream: int):
        """Enqueue the batched factorisation on `stream`; `ptrs` from pointer_array()."""
        self.lib.cusolverDnSetStream(self.handle, ctypes.c_void_p(stream))
        fill = 0 if uplo == "L" else 1              # CUBLAS_FILL_MODE_LOWER / UPPER
        st = getattr(self.lib, _FUNCS[dtype])(self.handle, fill, n, ctypes.c_void_p(ptrs.data_ptr()), lda,
                                              ctypes.c_void_p(info_ptr), batch)
        if st != 0:
            raise RuntimeError(f"{_FUNCS[dtype]} failed: status {st}")

    def close(self):
        if self.handle:
            self.lib.cusolverDnDestroy(self.handle)
            self.handle = ctypes.c_void_p()
