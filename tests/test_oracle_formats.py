"""Pins of the oracle's number formats (bf16, E4M3), independent of its code.

E4M3 is OCP FP8 e4m3fn (the dtype `float8_e4m3fn` of the Muse Spark attention
problem file's caches and q). The checks: brute-force nearest-code search over
all 256 codes, torch's own float8/bfloat16 casts, and round trips.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _e4m3_table():
    """Value of every finite E4M3 code from torch's cast (a library routine)."""
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


def test_e4m3_decode_matches_torch():
    codes, vals = _e4m3_table()
    ours = oracle.e4m3_value(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(ours[finite], vals[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(vals))
    assert np.isnan(vals).sum() == 2  # S.1111.111 only
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _brute_force_code(v: float, codes, vals) -> int:
    """Nearest finite code by exhaustive search; ties go to the even code;
    saturate beyond 448; keep the sign of zero."""
    if np.isnan(v):
        return 0x7F | (0x80 if np.signbit(v) else 0)
    if abs(v) >= 448.0:
        return 0x7E | (0x80 if v < 0 else 0)
    if v == 0.0:
        return 0x80 if np.signbit(v) else 0x00
    sign = 0x80 if v < 0 else 0
    a = Fraction(abs(v))
    best, best_d = None, None
    for c in range(0x00, 0x7F):  # non-negative finite codes
        d = abs(Fraction(vals[c]) - a)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | sign


def test_e4m3_encode_exhaustive_over_bf16():
    """All 65536 bf16 patterns: the oracle's encoder equals brute-force search."""
    codes, vals = _e4m3_table()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = oracle.bf16_value(bits)
    ours = oracle.e4m3_code(x)
    # brute force on the distinct magnitudes (the sign is handled separately)
    mags = np.unique(np.abs(x[~np.isnan(x)]))
    ref = {}
    for m in mags:
        ref[m] = _brute_force_code(float(m), codes, vals)
    for v, c in zip(x, ours):
        if np.isnan(v):
            assert c & 0x7F == 0x7F
            continue
        expect = ref[abs(v)] | (0x80 if np.signbit(v) else 0)
        if abs(v) == 0.0:
            expect = 0x80 if np.signbit(v) else 0x00
        assert c == expect, (v, c, expect)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (0.01, 1.0, 30.0)])
    x = x[np.abs(x) <= 448.0]
    ours = oracle.e4m3_code(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch casts float32; compare on inputs exactly representable in float32
    x32 = x.astype(np.float32).astype(np.float64)
    ours32 = oracle.e4m3_code(x32)
    assert np.array_equal(ours32, ref)
    assert ours.shape == ref.shape


def test_e4m3_round_trip_and_saturation():
    codes, vals = _e4m3_table()
    finite = ~np.isnan(vals)
    assert np.array_equal(oracle.e4m3_code(vals[finite]), codes[finite])
    big = np.array([448.0, 463.99, 464.0, 1e6, -500.0, np.inf, -np.inf])
    assert list(oracle.e4m3_code(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    # midpoints go to the even code: 1.0625 between 1.0 (0x38) and 1.125 (0x39)
    assert oracle.e4m3_code(np.array([1.0625, 1.1875]))[0] == 0x38
    assert oracle.e4m3_code(np.array([1.1875]))[0] == 0x3A  # between 0x39 and 0x3A -> even


def test_bf16_matches_torch():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(100000) * s for s in (1e-30, 1e-3, 1.0, 1e4)])
    x32 = x.astype(np.float32)
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # exact midpoints
    x32 = np.concatenate([x32, ties, -ties])
    ours = oracle.bf16_bits(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_from_double_is_single_rounding():
    """double -> bf16 rounds once: compare with exact rational nearest-even."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal(3000) * 3
    ours = oracle.bf16_value(oracle.bf16_bits(x))
    for v, r in zip(x, ours):
        # neighbours on the bf16 grid around v
        lo32 = np.float32(v)
        bits = int(np.array(lo32).view(np.uint32)) & 0xFFFF0000
        cand = []
        for db in (-1, 0, 1, 2):
            b = (bits + db * 0x10000) & 0xFFFFFFFF
            cand.append(float(np.array(b, dtype=np.uint32).view(np.float32)))
        fv = Fraction(v)
        best = min(cand, key=lambda c: (abs(Fraction(c) - fv),
                                        (int(np.array(np.float32(c)).view(np.uint32)) >> 16) & 1))
        assert r == best, (v, r, best)
