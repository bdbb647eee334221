"""Pins for the output-epilogue oracle."""
import numpy as np

from oracle import epilogue as ep
from synth.formats import to_bf16_bits


def test_no_shift_no_smooth_is_identity():
    x = np.random.default_rng(0).normal(size=(3, 4, 8))
    assert np.array_equal(ep.apply(x), x)


def test_shift_adds_and_smooth_multiplies_per_head_and_dim():
    x = np.zeros((2, 2, 4))
    shift = to_bf16_bits(np.arange(8, dtype=np.float32))          # exact in bf16
    smooth = to_bf16_bits(np.full(8, 2.0, np.float32))
    v = ep.apply(x + 1.0, shift, smooth)
    assert np.array_equal(v[0], (1.0 + np.arange(8).reshape(2, 4)) * 2.0)
    assert np.array_equal(v[1], v[0])


def test_int8_rounds_half_even_scales_and_clamps():
    v = np.array([0.5, 1.5, -0.5, 2.4999, 10.0, -10.0]) / 127.0
    q = ep.quantize_int8(v, in_scale=1.0, max_bound=127.0, min_bound=-127.0)
    assert q.tolist() == [0, 2, 0, 2, 10, -10]
    q2 = ep.quantize_int8(np.array([2.0, -3.0]), in_scale=1.0, max_bound=127.0, min_bound=-127.0)
    assert q2.tolist() == [127, -127]                                # saturation
    q3 = ep.quantize_int8(np.array([0.25]), in_scale=0.5, max_bound=100.0, min_bound=-100.0)
    assert q3.tolist() == [12]                                       # 0.25 * 100 * 0.5 = 12.5 -> 12
