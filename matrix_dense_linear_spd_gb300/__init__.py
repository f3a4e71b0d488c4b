"""Batched Cholesky factorisation (potrf) and SPD solves (posv, potrs) on GB300.

Thin ctypes binding over ``libbl.so`` (the C ABI in ``include/bl.h``). This module only
marshals arguments: every step of the computation runs in the library's CUDA kernels. There is
no CPU fallback: the first call raises ImportError if the library has not been built.

Tensor conventions: a batch of matrices is a tensor of shape (batch, n, n) whose matrices are
column-major, i.e. ``A.stride(-2) == 1``; ``A.stride(-1)`` is the leading dimension and
``A.stride(0)`` the item stride. ``colmajor(t)`` converts a row-major tensor into that layout.
Right-hand sides are (batch, n, nrhs), also with ``stride(-2) == 1``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbl.so")

BL_LOWER, BL_UPPER = 0, 1
BL_F32, BL_F64, BL_C64, BL_C128 = 0, 1, 2, 3
DTYPE_CODES = {"f32": BL_F32, "f64": BL_F64, "c64": BL_C64, "c128": BL_C128}
STATUS = {0: "success", 1: "invalid argument", 2: "no route", 3: "CUDA error", 4: "internal error"}

EXPORTED = ("bl_potrf", "bl_posv", "bl_potrs", "bl_status_string", "bl_last_error", "bl_last_choice",
            "bl_version", "bl_set_route", "bl_num_routes", "bl_route_name", "bl_route_capacity",
            "bl_select_debug", "bl_debug_tc_tile_f32", "bl_debug_peak")


class BLError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m matrix_dense_linear_spd_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, i32p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.bl_potrf.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, vp, i64, i64, i32p, vp]
    lib.bl_posv.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, vp, i64, i64, vp, i64, i64, i32p, vp]
    lib.bl_potrs.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp]
    for f in ("bl_potrf", "bl_posv", "bl_potrs", "bl_set_route"):
        getattr(lib, f).restype = ctypes.c_int
    lib.bl_status_string.argtypes = [ctypes.c_int]
    lib.bl_status_string.restype = ctypes.c_char_p
    lib.bl_last_error.restype = ctypes.c_char_p
    lib.bl_last_choice.restype = ctypes.c_char_p
    lib.bl_version.restype = ctypes.c_int
    lib.bl_set_route.argtypes = [ctypes.c_char_p, ctypes.c_char_p]
    lib.bl_num_routes.argtypes = [ctypes.c_int]
    lib.bl_num_routes.restype = ctypes.c_int
    lib.bl_route_name.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.bl_route_name.restype = ctypes.c_char_p
    lib.bl_route_capacity.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.bl_route_capacity.restype = ctypes.c_int
    lib.bl_select_debug.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, i64,
                                    ctypes.c_char_p, i64]
    lib.bl_select_debug.restype = ctypes.c_char_p
    lib.bl_debug_tc_tile_f32.argtypes = [vp, vp, vp, vp, vp]
    lib.bl_debug_tc_tile_f32.restype = ctypes.c_int
    lib.bl_debug_peak.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.POINTER(ctypes.c_double), vp]
    lib.bl_debug_peak.restype = ctypes.c_int
    return lib


_lib = None


def get_lib():
    """The loaded libbl.so (loaded on first use; raises ImportError if it is missing)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(status: int):
    if status != 0:
        raise BLError(status, get_lib().bl_last_error().decode())


def _uplo(u) -> int:
    if u in ("L", "l", BL_LOWER, "lower"):
        return BL_LOWER
    if u in ("U", "u", BL_UPPER, "upper"):
        return BL_UPPER
    raise ValueError(f"uplo must be 'L' or 'U', not {u!r}")


# ------------------------------------------------------------------ raw-pointer entry points

def potrf_ptr(uplo, dtype: int, n: int, batch: int, A: int, lda: int, stride_a: int, info: int,
              stream: int = 0) -> None:
    _check(get_lib().bl_potrf(_uplo(uplo), dtype, n, batch, A, lda, stride_a, info, stream))


def posv_ptr(uplo, dtype: int, n: int, nrhs: int, batch: int, A: int, lda: int, stride_a: int,
             B: int, ldb: int, stride_b: int, info: int, stream: int = 0) -> None:
    _check(get_lib().bl_posv(_uplo(uplo), dtype, n, nrhs, batch, A, lda, stride_a, B, ldb, stride_b, info,
                       stream))


def potrs_ptr(uplo, dtype: int, n: int, nrhs: int, batch: int, A: int, lda: int, stride_a: int,
              B: int, ldb: int, stride_b: int, stream: int = 0) -> None:
    _check(get_lib().bl_potrs(_uplo(uplo), dtype, n, nrhs, batch, A, lda, stride_a, B, ldb, stride_b, stream))


def set_route(op: str, spelling: str | None) -> None:
    """Pin the kernel variant for op ('potrf', 'posv', 'potrs') on this thread; None clears."""
    _check(get_lib().bl_set_route(op.encode(), spelling.encode() if spelling else None))


def routes(dtype: str):
    """[(spelling, capacity, rhs_per_pass)] for every compiled variant of dtype."""
    lib = get_lib()
    code = DTYPE_CODES[dtype]
    out = []
    for i in range(lib.bl_num_routes(code)):
        rp = ctypes.c_int(0)
        cap = lib.bl_route_capacity(code, i, ctypes.byref(rp))
        out.append((lib.bl_route_name(code, i).decode(), cap, rp.value))
    return out


def select_debug(op: str, dtype: str, uplo: str, n: int, nrhs: int = 0, batch: int = 1,
                 devkey: str = "sm_103", smem_optin: int = 232448) -> str:
    """The variant `op` would choose on a synthetic device (host logic only, no GPU needed)."""
    code = {"potrf": 0, "posv": 1, "potrs": 2}[op]
    return get_lib().bl_select_debug(code, DTYPE_CODES[dtype], _uplo(uplo), n, nrhs, batch,
                                     devkey.encode(), smem_optin).decode()


def last_choice() -> str:
    return get_lib().bl_last_choice().decode()


# ------------------------------------------------------------------ torch-tensor entry points

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    codes = {torch.float32: BL_F32, torch.float64: BL_F64, torch.complex64: BL_C64,
             torch.complex128: BL_C128}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _batch_view(M, name):
    """(batch, rows, cols) view of a column-major tensor; returns (view, ld, stride)."""
    if M.dim() == 2:
        M = M.unsqueeze(0)
    if M.dim() != 3:
        raise ValueError(f"{name} must be (rows, cols) or (batch, rows, cols)")
    if not M.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if M.shape[-2] > 1 and M.stride(-2) != 1:
        raise ValueError(f"{name} must be column-major (stride(-2) == 1); see colmajor()")
    ld = M.stride(-1) if M.shape[-1] > 1 else max(M.shape[-2], 1)
    stride = M.stride(0) if M.shape[0] > 1 else ld * M.shape[-1]
    return M, ld, stride


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def colmajor(t):
    """Copy of a (batch, rows, cols) tensor stored column-major (same logical values)."""
    return t.transpose(-1, -2).contiguous().transpose(-1, -2)


def colmajor_empty(batch: int, rows: int, cols: int, dtype, device="cuda"):
    torch = _torch()
    return torch.empty(batch, cols, rows, dtype=dtype, device=device).transpose(-1, -2)


def potrf(A, uplo="L", info=None, stream=None):
    """Factor the batch A in place (referenced triangle only). Returns the int32 info tensor."""
    torch = _torch()
    A3, lda, sa = _batch_view(A, "A")
    batch, n, n2 = A3.shape
    if n != n2:
        raise ValueError("A must be square")
    if info is None:
        info = torch.empty(batch, dtype=torch.int32, device=A3.device)
    potrf_ptr(uplo, _dtype_code(A3), n, batch, A3.data_ptr(), lda, sa, info.data_ptr(), _stream(stream))
    return info


def posv(A, B, uplo="L", info=None, stream=None):
    """Factor A and solve A X = B in place (A <- factor, B <- X). Returns the info tensor."""
    torch = _torch()
    A3, lda, sa = _batch_view(A, "A")
    B3, ldb, sb = _batch_view(B, "B")
    batch, n, _ = A3.shape
    if B3.shape[0] != batch or B3.shape[1] != n or B3.dtype != A3.dtype:
        raise ValueError("B must be (batch, n, nrhs) of A's dtype")
    if info is None:
        info = torch.empty(batch, dtype=torch.int32, device=A3.device)
    posv_ptr(uplo, _dtype_code(A3), n, B3.shape[2], batch, A3.data_ptr(), lda, sa, B3.data_ptr(), ldb,
             sb, info.data_ptr(), _stream(stream))
    return info


def potrs(A, B, uplo="L", stream=None):
    """Solve A X = B with the factor stored in A's `uplo` triangle; B <- X."""
    A3, lda, sa = _batch_view(A, "A")
    B3, ldb, sb = _batch_view(B, "B")
    batch, n, _ = A3.shape
    if B3.shape[0] != batch or B3.shape[1] != n or B3.dtype != A3.dtype:
        raise ValueError("B must be (batch, n, nrhs) of A's dtype")
    potrs_ptr(uplo, _dtype_code(A3), n, B3.shape[2], batch, A3.data_ptr(), lda, sa, B3.data_ptr(), ldb,
              sb, _stream(stream))
