"""Pins for the oracle's element formats (CPU only).

Each encoder is checked against an exhaustive brute-force search written
independently here: exact integer arithmetic (values scaled by 2**200), the
nearest grid point by scanning the whole grid, ties to the even code.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F

SCALE = 1 << 200


def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_f32(bits)
    fin = np.isfinite(v)
    return bits[fin], v[fin]


def _brute_nearest_codes(values, grid_vals, sign_bit):
    grid = [int(Fraction(float(g)) * SCALE) for g in grid_vals]
    out = np.empty(len(values), dtype=np.uint8)
    for n, x in enumerate(values):
        xi = int(Fraction(float(x)) * SCALE)
        a = abs(xi)
        best, bi = None, 0
        for i, g in enumerate(grid):
            d = abs(a - g)
            if best is None or d < best or (d == best and i % 2 == 0):
                best, bi = d, i
        neg = xi < 0 or (xi == 0 and np.signbit(x))
        out[n] = bi | (sign_bit if neg else 0)
    return out


def test_e2m1_grid_is_the_pages_grid():
    # The E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} (1 sign, 2 exponent,
    # 1 mantissa bit, bias 1) written out from the bit fields.
    vals = []
    for code in range(8):
        e, m = code >> 1, code & 1
        vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    assert vals == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert np.array_equal(F.E2M1_GRID, vals)


def test_e4m3_range():
    assert F.E4M3_GRID[-1] == 448.0                  # largest finite, code 0x7E
    assert F.E4M3_GRID[1] == 2.0 ** -9               # smallest subnormal
    assert F.E4M3_GRID[8] == 2.0 ** -6               # smallest normal
    assert np.all(np.diff(F.E4M3_GRID) > 0)
    assert np.isnan(F.e4m3_decode(0x7F)) and np.isnan(F.e4m3_decode(0xFF))
    assert len(F.E4M3_GRID) == 127


def test_e8m0_range():
    assert F.e8m0_decode(127) == 1.0
    assert F.e8m0_decode(0) == 2.0 ** -127
    assert F.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(F.e8m0_decode(255))


def test_e2m1_encode_exhaustive_bf16():
    _, v = _all_finite_bf16()
    got = F.e2m1_encode(v)
    ref = _brute_nearest_codes(v, F.E2M1_GRID, 0x8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_exhaustive_bf16():
    _, v = _all_finite_bf16()
    got = F.e4m3_encode(v)
    ref = _brute_nearest_codes(v, F.E4M3_GRID, 0x80)
    assert np.array_equal(got, ref)


def test_e4m3_encode_fp32_sample_vs_brute():
    # fp32 inputs (the NVFP4 block-scale path encodes fp32 values)
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    v = np.concatenate([v, (rng.standard_normal(4000) * 100).astype(np.float32)])
    assert np.array_equal(F.e4m3_encode(v), _brute_nearest_codes(v, F.E4M3_GRID, 0x80))


def test_e2m1_ties():
    # ties to even code: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    t = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.01, 100.0])
    assert list(F.e2m1_decode(F.e2m1_encode(t))) == [0, 1, 1, 2, 2, 4, 4, 6, 6]
    assert list(F.e2m1_decode(F.e2m1_encode(-t))) == [0, -1, -1, -2, -2, -4, -4, -6, -6]


def test_roundtrip_every_code():
    for c in range(16):
        assert F.e2m1_encode(F.e2m1_decode(np.array([c])))[0] == c
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert F.e4m3_encode(F.e4m3_decode(np.array([c])))[0] == c


def test_negative_zero_keeps_sign():
    assert F.e2m1_encode(np.array([-0.1]))[0] == 0x8
    assert F.e4m3_encode(np.array([-1e-9]))[0] == 0x80
    assert F.e4m3_encode(np.array([-0.0]))[0] == 0x80


def test_e8m0_rule_exhaustive_bf16():
    """Smallest e with a <= 448 * 2**e, found by exact search, for every finite
    positive bf16 amax; the block max never clips after scaling."""
    bits, v = _all_finite_bf16()
    pos = v > 0
    a = v[pos].astype(np.float64)
    got = F.e8m0_exponent_for_amax(a)
    # independent search in exact integer arithmetic: a = num / 2**200, so
    # a <= 448 * 2**e  <=>  num <= 448 * 2**(e + 200)
    for ai, ei in zip(a[::7], got[::7]):
        num = int(Fraction(float(ai)) * SCALE)
        e = -127
        while e < 127 and num > 448 * 2 ** (e + 200):
            e += 1
        assert e == ei
    # no clipping: a * 2**-e <= 448 exactly, and e is minimal (or clamped)
    assert np.all(a * np.ldexp(1.0, -got) <= 448.0)
    lower = a * np.ldexp(1.0, -(got - 1))
    assert np.all((lower > 448.0) | (got == -127))
    # closed form for a = 1.f * 2**p:  e = p - 8 + [1.f > 1.75]
    m, p = np.frexp(a)
    closed = (p - 1) - 8 + ((2 * m) > 1.75)
    assert np.array_equal(np.clip(closed, -127, 127), got)
    # zero amax gives the clamp value
    assert F.e8m0_exponent_for_amax(np.array([0.0]))[0] == -127


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9, -3.14159,
                  2.0 ** -130, 1.0 + 3 * 2 ** -8])
    got = F.bf16_round(x)
    assert got[0] == 1.0
    assert got[1] == 1.0                  # halfway, ties to the even mantissa
    assert got[2] == 1.0 + 2 ** -7        # above halfway
    assert got[3] == 1.0                  # below halfway
    assert got[4] == -3.140625
    assert got[5] == 2.0 ** -130          # bf16 subnormal, exact
    assert got[6] == 1.0 + 2 ** -6        # halfway, rounds up to the even mantissa
    # against torch's bf16 conversion of fp32 inputs that are exact in fp32
    import torch
    v = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16_round(v.astype(np.float64)), ref)
