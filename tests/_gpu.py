"""Helpers for the GPU parity tests: run the library through its C ABI on seeded synthetic
inputs and compare with the CPU oracle, element by element.

Tolerances (stated in the library's acceptance criteria for inputs with condition number
<= 1e3): per-item relative Frobenius error of the factor over the referenced triangle
<= 2e-4 (f32, c64) / 1e-11 (f64, c128); posv solution <= 1e-3 / 1e-10; info bit-exact.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
import synth

TOL_F = {"f32": 2e-4, "c64": 2e-4, "f64": 1e-11, "c128": 1e-11}
TOL_X = {"f32": 1e-3, "c64": 1e-3, "f64": 1e-10, "c128": 1e-10}
THREADS = max(1, min(32, os.cpu_count() or 1))


def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        import pytest
        pytest.skip("no CUDA device")
    return torch


def lib():
    import matrix_dense_linear_spd_gb300 as bl
    return bl


def dev(buf):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(buf)).cuda()


def call_potrf(A, uplo, dtype, ld=None, stride=None, fill=0, route=None):
    """Run bl_potrf on logical matrices A (batch, n, n). Returns (input buffer, output buffer,
    info, ld, stride)."""
    torch = torch_cuda()
    bl = lib()
    batch, n, _ = A.shape
    ld = n if ld is None else ld
    stride = ld * n if stride is None else stride
    buf = synth.to_colmajor(A, ld, stride, fill)
    d = dev(buf)
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    if route:
        bl.set_route("potrf", route)
    try:
        bl.potrf_ptr(uplo, bl.DTYPE_CODES[dtype], n, batch, d.data_ptr(), ld, stride, info.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    finally:
        if route:
            bl.set_route("potrf", None)
    torch.cuda.synchronize()
    return buf, d.cpu().numpy(), info.cpu().numpy(), ld, stride


def call_posv(A, B, uplo, dtype, ld=None, stride=None, ldb=None, stride_b=None, fill=0, route=None,
              op="posv", info_init=-7):
    torch = torch_cuda()
    bl = lib()
    batch, n, _ = A.shape
    nrhs = B.shape[-1]
    ld = n if ld is None else ld
    stride = ld * n if stride is None else stride
    ldb = n if ldb is None else ldb
    stride_b = ldb * nrhs if stride_b is None else stride_b
    abuf = synth.to_colmajor(A, ld, stride, fill)
    bbuf = synth.to_colmajor(B, ldb, stride_b, fill)
    da, db = dev(abuf), dev(bbuf)
    info = torch.full((batch,), info_init, dtype=torch.int32, device="cuda")
    if route:
        bl.set_route(op, route)
    try:
        s = torch.cuda.current_stream().cuda_stream
        if op == "posv":
            bl.posv_ptr(uplo, bl.DTYPE_CODES[dtype], n, nrhs, batch, da.data_ptr(), ld, stride, db.data_ptr(),
                        ldb, stride_b, info.data_ptr(), s)
        else:
            bl.potrs_ptr(uplo, bl.DTYPE_CODES[dtype], n, nrhs, batch, da.data_ptr(), ld, stride, db.data_ptr(),
                         ldb, stride_b, s)
    finally:
        if route:
            bl.set_route(op, None)
    torch.cuda.synchronize()
    return abuf, da.cpu().numpy(), bbuf, db.cpu().numpy(), info.cpu().numpy()


def tri_mask(n, uplo):
    return np.tril(np.ones((n, n), bool)) if uplo == "L" else np.triu(np.ones((n, n), bool))


def factor_errors(out_buf, ref, info, n, batch, ld, stride, uplo, items=None):
    """Per-item relative Frobenius error of the GPU factor against the oracle's, over the
    referenced triangle of the leading (info-1) block (whole matrix on success)."""
    F = synth.from_colmajor(out_buf, n, n, batch, ld, stride)
    mask = tri_mask(n, uplo)
    items = range(batch) if items is None else items
    errs = []
    for k, b in enumerate(items):
        m = n if info[b] == 0 else int(info[b]) - 1
        if m == 0:
            errs.append(0.0)
            continue
        r = ref[k][:m, :m]
        g = F[b][:m, :m].astype(r.dtype)
        msk = mask[:m, :m]
        diff = np.where(msk, g - r, 0)
        num = np.sqrt(np.sum(np.abs(diff) ** 2))
        den = np.sqrt(np.sum(np.abs(np.where(msk, r, 0)) ** 2))
        errs.append(float(num / den) if den > 0 else float(num))
    return np.array(errs)


def other_triangle_unchanged(in_buf, out_buf, n, batch, ld, stride, uplo):
    """Bytes outside the referenced triangle (other triangle, ld padding and item gaps) are
    bit-identical after the call."""
    a = synth.from_colmajor(in_buf, n, n, batch, ld, stride)
    b = synth.from_colmajor(out_buf, n, n, batch, ld, stride)
    other = ~tri_mask(n, uplo)
    same_tri = np.array_equal(np.ascontiguousarray(a[:, other]).view(np.uint8),
                              np.ascontiguousarray(b[:, other]).view(np.uint8))
    # gaps between columns / items
    idx = np.zeros(in_buf.size, bool)
    for c in range(n):
        for_items = np.arange(batch)[:, None] * stride + c * ld + np.arange(n)[None, :]
        idx[for_items.ravel()] = True
    same_gap = np.array_equal(np.ascontiguousarray(in_buf[~idx]).view(np.uint8),
                              np.ascontiguousarray(out_buf[~idx]).view(np.uint8))
    return same_tri and same_gap


def solution_errors(X_gpu, X_ref):
    errs = []
    for b in range(X_ref.shape[0]):
        r = X_ref[b]
        g = X_gpu[b].astype(r.dtype)
        errs.append(float(np.sqrt(np.sum(np.abs(g - r) ** 2)) / np.sqrt(np.sum(np.abs(r) ** 2))))
    return np.array(errs)
