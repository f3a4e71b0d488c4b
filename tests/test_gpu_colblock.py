"""GPU parity of the column-block tensor-core kernel (blocked:nb=32:tc=2, f32 potrf, n <= 512)
against the CPU oracle, pinned through the C ABI.

The kernel keeps a block of 128 columns as f32 accumulators in tensor memory and factors it 32
columns at a time, so the cases below put the order, the planted failures and the layout on
every boundary it has: slice (32), block (128), row tile (128), and ragged ends.
"""
import numpy as np
import pytest

import synth
from _gpu import TOL_F, call_potrf, lib, torch_cuda
from test_gpu_parity import _check_potrf

pytestmark = pytest.mark.gpu

ROUTE = "blocked:nb=32:tc=2"
ORDERS = [1, 2, 7, 31, 32, 33, 63, 64, 100, 127, 128, 129, 160, 191, 200, 255, 256, 257, 300, 383, 384, 385, 450,
          479, 511, 512]


def _spd(rng, n, batch):
    return synth.spd_bbt(rng, n, batch, "f32")


@pytest.mark.parametrize("uplo", ["L", "U"])
def test_orders_across_slice_block_and_tile_edges(uplo):
    rng = np.random.default_rng(41)
    for n in ORDERS:
        _check_potrf(_spd(rng, n, 3), uplo, "f32", route=ROUTE)


def test_haar_spectrum_inputs():
    """A = Q diag(lambda) Q^T with lambda log-uniform in [1, 1e3] (the conditioned construction)."""
    rng = np.random.default_rng(43)
    for n in (96, 200, 512):
        A = synth.spd_haar(rng, n, 2, "f32")
        for uplo in "LU":
            _check_potrf(A, uplo, "f32", route=ROUTE)


@pytest.mark.parametrize("uplo", ["L", "U"])
def test_planted_failures_in_every_slice_and_block(uplo):
    """A(k,k) = -1 fails exactly at column k (info = k+1), wherever k falls; a NaN pivot too;
    two planted failures report the first."""
    rng = np.random.default_rng(47)
    n = 300
    ks = [0, 5, 31, 32, 63, 100, 127, 128, 129, 200, 255, 256, 299]
    A = _spd(rng, n, len(ks) + 3)
    expect = np.zeros(len(ks) + 3, np.int32)
    for b, k in enumerate(ks):
        A[b, k, k] = -1
        expect[b] = k + 1
    A[len(ks), 140, 140] = np.nan
    expect[len(ks)] = 141
    A[len(ks) + 1, 250, 250] = -1
    A[len(ks) + 1, 70, 70] = -1
    expect[len(ks) + 1] = 71
    _check_potrf(A, uplo, "f32", expect_info=expect, route=ROUTE)


@pytest.mark.parametrize("uplo", ["L", "U"])
def test_padded_layout_is_bit_identical_and_gaps_untouched(uplo):
    """ld = n + 7, stride = ld*n + 13 with NaN in the padding and gaps: same bits as the natural
    layout, padding and gaps unchanged, other triangle unchanged (checked inside)."""
    rng = np.random.default_rng(53)
    for n in (77, 300):
        A = _spd(rng, n, 2)
        nat, _, _ = _check_potrf(A, uplo, "f32", route=ROUTE)
        pad, _, _ = _check_potrf(A, uplo, "f32", ld=n + 7, stride=(n + 7) * n + 13, fill=np.nan, route=ROUTE)
        Fn = synth.from_colmajor(nat, n, n, 2)
        Fp = synth.from_colmajor(pad, n, n, 2, n + 7, (n + 7) * n + 13)
        assert np.array_equal(Fn.view(np.uint32), Fp.view(np.uint32))


def test_other_triangle_poison_has_no_effect():
    """NaN in the other triangle changes no bit of the factor."""
    rng = np.random.default_rng(59)
    n = 260
    A = _spd(rng, n, 2)
    clean, _, _ = _check_potrf(A, "L", "f32", route=ROUTE)
    P = A.copy()
    P[:, np.triu(np.ones((n, n), bool), 1)] = np.nan
    _, out, info, _, _ = call_potrf(P, "L", "f32", route=ROUTE)
    assert not info.any()
    low = np.tril(np.ones((n, n), bool))
    a = synth.from_colmajor(clean, n, n, 2)[:, low]
    b = synth.from_colmajor(out, n, n, 2)[:, low]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_batch_larger_than_the_grid_wave_and_identical_items():
    """Many CTAs (more than one per SM) on identical items give identical bits."""
    rng = np.random.default_rng(61)
    n = 256
    one = _spd(rng, n, 1)
    A = np.repeat(one, 400, axis=0)
    _, out, info, _, _ = call_potrf(A, "L", "f32", route=ROUTE)
    assert not info.any()
    F = synth.from_colmajor(out, n, n, 400).view(np.uint32)
    assert (F == F[0]).all()


def test_refuses_orders_above_512_and_solves():
    bl = lib()
    torch = torch_cuda()
    d = torch.zeros(513 * 513, dtype=torch.float32, device="cuda")
    info = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    bl.set_route("potrf", ROUTE)
    try:
        with pytest.raises(bl.BLError):
            bl.potrf_ptr("L", bl.BL_F32, 513, 1, d.data_ptr(), 513, 513 * 513, info.data_ptr(), s)
    finally:
        bl.set_route("potrf", None)
    bl.set_route("posv", ROUTE)
    try:
        with pytest.raises(bl.BLError):
            bl.posv_ptr("L", bl.BL_F32, 64, 1, 1, d.data_ptr(), 64, 64 * 64, d.data_ptr(), 64, 64, info.data_ptr(), s)
    finally:
        bl.set_route("posv", None)
    torch.cuda.synchronize()
    assert TOL_F["f32"] == 2e-4
