"""The seeded input generators: the threaded C draws (synth/csrc/synth_host.c)
against the numpy statement of the same counter formulas in synth.rng."""
import numpy as np
import pytest

from synth import rng


def _have_lib():
    return rng._host_lib() is not None


@pytest.mark.skipif(not _have_lib(), reason="host generator library not built")
@pytest.mark.parametrize("seed,stream,start,n", [(1, 3, 0, 1000), (5, 4, 123456789, 300000),
                                                 (2 ** 40 + 7, 11, 2 ** 33, 70000)])
def test_c_normal_matches_numpy_definition(seed, stream, start, n):
    idx = np.arange(start, start + n, dtype=np.uint64)
    c = rng.normal(seed, stream, idx)
    ref = rng.normal_np(seed, stream, idx)
    # the two libraries' log1p / cos may differ in the last bits only
    assert np.all(np.abs(c - ref) <= 4 * np.spacing(np.abs(ref)) + 1e-300)
    assert np.mean(c == ref) > 0.5


@pytest.mark.skipif(not _have_lib(), reason="host generator library not built")
@pytest.mark.parametrize("lo,hi", [(-127, 127), (-128, 127), (-3, 5), (0, 0)])
def test_c_uniform_int8_bytes_match_numpy_definition(lo, hi):
    start, n = 987654321, 1 << 21
    c = rng.uniform_i8_bytes(7, 4, start, n, lo, hi)
    ref = np.asarray(rng.uniform_int(7, 4, np.arange(start, start + n, dtype=np.uint64), lo, hi))
    assert np.array_equal(c, ref.astype(np.int8).view(np.uint8))


def test_normal_falls_back_for_scattered_counters():
    idx = np.array([5, 1, 9, 2], dtype=np.uint64)
    assert np.array_equal(rng.normal(3, 2, idx), rng.normal_np(3, 2, idx))


def test_normal_draws_are_standard():
    x = rng.normal(9, 1, np.arange(1 << 20, dtype=np.uint64))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
