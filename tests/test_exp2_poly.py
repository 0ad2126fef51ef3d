"""CPU checks of the FMA-pipe 2^x that the attention softmax uses for one score pair in four:
the coefficients compiled into the kernel are the Remez fit of exp2_poly.fit() rounded to fp32,
the fit equioscillates, and the kernel's fp32 arithmetic (modelled bit for bit) stays within its
stated relative error of the exact 2^x over the range the softmax feeds it."""
import os
import re

import numpy as np

from streaming_causal_video_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kernel_coefficients():
    text = open(os.path.join(ROOT, "streaming_causal_video_gb300", "csrc", "ptx.cuh")).read()
    got = dict(re.findall(r"constexpr float kExp2C(\d) = ([0-9.eE+-]+)f;", text))
    assert sorted(got) == ["0", "1", "2", "3"]
    return [np.float32(float(got[str(k)])) for k in range(4)]


def test_kernel_coefficients_are_the_remez_fit():
    c, err = exp2_poly.fit(3)
    assert err < 7.5e-5
    assert kernel_coefficients() == [np.float32(v) for v in c]


def test_fit_equioscillates_and_beats_taylor():
    c, err = exp2_poly.fit(3)
    xs = np.linspace(0, 1, 200001)
    e = np.polyval(np.array(c)[::-1], xs) / np.exp2(xs) - 1
    # minimax: the error reaches +-err at both ends and alternates in sign 5 times
    assert abs(abs(e[0]) - err) < 1e-7 and abs(abs(e[-1]) - err) < 1e-7
    assert len(np.flatnonzero(np.diff(np.sign(e)) != 0)) == 4
    taylor = [1.0, np.log(2), np.log(2) ** 2 / 2, np.log(2) ** 3 / 6]
    et = np.polyval(np.array(taylor)[::-1], xs) / np.exp2(xs) - 1
    assert np.abs(et).max() > 10 * err


def test_kernel_arithmetic_relative_error_over_the_softmax_range():
    c32 = kernel_coefficients()
    x = np.concatenate([np.linspace(-125, 8, 3_000_001), -np.arange(0, 126, dtype=np.float64)]).astype(np.float32)
    y = exp2_poly.model_f32(x, c32).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() <= 7.6e-5, (rel.max(), x[rel.argmax()])
    # integers: f = 0 exactly, so 2^n * c0
    n = np.arange(-125, 9, dtype=np.float32)
    np.testing.assert_array_equal(exp2_poly.model_f32(n, c32), (np.float32(c32[0]) * np.exp2(n)).astype(np.float32))


def test_far_below_the_range_is_tiny_positive_never_nan():
    c32 = kernel_coefficients()
    x = np.array([-np.inf, -1e30, -1000, -127, -126.5, -126], np.float32)
    y = exp2_poly.model_f32(x, c32)
    assert np.all(np.isfinite(y)) and np.all(y > 0) and np.all(y <= np.float32(2.0 ** -125))
