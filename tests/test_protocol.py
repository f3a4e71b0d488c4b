"""Host-side tests of the measurement protocol's bookkeeping (no GPU): how many pristine copies a
back-to-back chunk takes, and the statistics the benchmark reports."""
import pytest

from matrix_dense_linear_spd_gb300 import protocol as P

L2 = 129 << 20


def test_copies_exceed_four_times_l2_when_the_batch_allows():
    item = 64 << 20                                     # f32 n=32 b16384
    r = P.copies_per_chunk(item, L2, steps=200)
    assert r == 20 and r * item > 4 * L2


def test_large_items_take_few_copies_and_respect_the_memory_cap():
    item = 2 << 30                                      # f64 n=512 b1024
    r = P.copies_per_chunk(item, L2, steps=200)
    assert r == 2 and r * item <= 4 << 30
    assert P.copies_per_chunk(8 << 30, L2, steps=200) == 1      # never zero


def test_copies_never_exceed_the_steps():
    assert P.copies_per_chunk(33 << 10, L2, steps=5) == 5       # tiny items: as many as steps


def test_stats():
    st = P.stats([1.0, 2.0, 3.0, 4.0])
    assert st["median"] == 2.5 and st["mean"] == 2.5 and st["n"] == 4
    assert st["rel_sd"] == pytest.approx((1.25 ** 0.5) / 2.5)
    assert P.stats([5.0])["rel_sd"] == 0.0
