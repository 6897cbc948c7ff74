"""Pins of the oracle's RoPE table (`_cos_sin` of the Muse Spark attention
problem file) against high-precision arithmetic (mpmath), not against itself.

The reading: inv_freq[i] = f32(1 / f32(theta^(2i/64))), angle = f32(f32(pos) *
inv_freq[i]), cos/sin = f32 of the exact value — each float32 result the
correctly rounded value of its exact operation.
"""
import numpy as np
import pytest

import oracle

mpmath = pytest.importorskip("mpmath")
mpmath.mp.prec = 200


def _round_f32(x) -> np.float32:
    """Correctly rounded float32 of an mpmath number (nearest, ties to even)."""
    guess = np.float32(float(x))
    cands = [np.nextafter(guess, np.float32(-np.inf)), guess, np.nextafter(guess, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(mpmath.mpf(float(c)) - x),
                                     int(np.array(c).view(np.uint32)) & 1))
    return np.float32(best)


@pytest.mark.parametrize("theta", [5e5, 1e4])
def test_inv_freq_correctly_rounded(theta):
    inv = oracle.rope_inv_freq(theta)
    th = mpmath.mpf(float(np.float32(theta)))
    for i in range(32):
        e = mpmath.mpf(2 * i) / 64
        pw = _round_f32(th ** e)
        expect = _round_f32(1 / mpmath.mpf(float(pw)))
        assert inv[i] == expect, (i, inv[i], expect)
    assert inv[0] == 1.0  # theta^0


@pytest.mark.parametrize("pos", [0, 1, 7, 100, 2047, 8191, 131072, (1 << 21) - 1])
def test_cos_sin_rows(pos):
    theta = 5e5
    c, s = oracle.rope_row(theta, pos)
    inv = oracle.rope_inv_freq(theta)
    for i in range(32):
        ang = np.float32(np.float32(pos) * inv[i])  # one float32 rounding of the product
        a = mpmath.mpf(float(ang))
        assert c[i] == _round_f32(mpmath.cos(a)), (pos, i)
        assert s[i] == _round_f32(mpmath.sin(a)), (pos, i)
    if pos == 0:
        assert np.all(c == 1.0) and np.all(s == 0.0)


def test_angles_decrease_with_pair_index():
    inv = oracle.rope_inv_freq(5e5)
    assert np.all(np.diff(inv) < 0) and inv[-1] > 0
