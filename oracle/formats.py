"""Element formats: E2M1, E4M3 (fn), E8M0 and bf16 (oracle; test infrastructure).

"Towards Blackwell-native 8-bit and 4-bit RL", section "Format background",
names the formats: MXFP8 = E4M3 elements with an E8M0 block scale, NVFP4 =
E2M1 elements with an E4M3 block scale.  The grids below are those formats'
standard definitions:

* E2M1: magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, codes 0..7, sign in bit 3.
* E4M3 (fn): exponent bias 7, subnormals k * 2**-9, largest finite 448
  (code 0x7E); 0x7F / 0xFF are NaN; no infinity.
* E8M0: value 2**(b - 127) for b in 0..254; 0xFF is NaN.

Every encoder rounds to the nearest point of the grid, ties to the even code,
and saturates to the largest finite magnitude.  A negative value that rounds
to zero keeps its sign bit.  All comparisons are exact: inputs are fp32 or
bf16 values held in fp64, and every difference taken below is exactly
representable in fp64.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- bf16 / fp32


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns with ONE round-to-nearest-even step.

    The value is rounded straight from fp64 onto the bf16 grid (8 significant
    bits), not through fp32, so no double rounding occurs.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 normal numbers carry 8 significant bits: scale m to [128, 256)
    q = np.rint(m * 256.0)                  # rint = round half to even
    y = np.ldexp(q, e - 8)
    # bf16 subnormals: spacing 2**-133 below 2**-126
    small = np.abs(x) < 2.0 ** -126
    if np.any(small):
        ys = np.rint(x[small] * 2.0 ** 133) * 2.0 ** -133
        y = y.copy()
        y[small] = ys
    y32 = y.astype(np.float32)              # exact: y is on the bf16 grid
    return (y32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value, returned as fp64."""
    return bf16_bits_to_f32(f64_to_bf16_bits(x)).astype(np.float64)


# ---------------------------------------------------------------- grids

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_value(code: int) -> float:
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0:
        return man * 2.0 ** -9
    return (1.0 + man / 8.0) * 2.0 ** (exp - 7)


# non-negative finite E4M3 values, codes 0x00 .. 0x7E (strictly increasing)
E4M3_GRID = np.array([_e4m3_value(c) for c in range(0x7F)])
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _encode_on_grid(x: np.ndarray, grid: np.ndarray, sign_bit: int) -> np.ndarray:
    """Nearest grid point, ties to the even code, saturating; sign bit kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = len(grid) - 1
    hi = np.searchsorted(grid, a, side="left")          # grid[hi-1] < a <= grid[hi]
    hi = np.clip(hi, 1, top)
    lo = hi - 1
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= grid[top], top, code)          # saturate
    code = np.where(a <= grid[0], 0, code)
    neg = np.signbit(x)
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Values -> E2M1 codes (uint8 in 0..15), RNE on the grid, satfinite."""
    return _encode_on_grid(x, E2M1_GRID, 0x8)


def e2m1_decode(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c).astype(np.int64)
    v = E2M1_GRID[c & 0x7]
    return np.where((c & 0x8) != 0, -v, v)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Values -> E4M3 (fn) codes, RNE on the grid, saturating to +-448."""
    return _encode_on_grid(x, E4M3_GRID, 0x80)


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c).astype(np.int64)
    mag = c & 0x7F
    v = np.where(mag == 0x7F, np.nan, E4M3_GRID[np.minimum(mag, 0x7E)])
    return np.where((c & 0x80) != 0, -v, v)


def e8m0_decode(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b).astype(np.int64)
    return np.where(b == 0xFF, np.nan, np.ldexp(1.0, b - 127))


def e8m0_exponent_for_amax(a: np.ndarray) -> np.ndarray:
    """Smallest integer e with a <= 448 * 2**e, clamped to [-127, 127].

    This is the MXFP8 "round the scale up to a power of two so that the block
    max never clips" rule written out: start from an estimate and correct it
    with exact comparisons against 448 * 2**e (exact in fp64).  a = 0 gives the
    clamp value -127.
    """
    a = np.asarray(a, dtype=np.float64)
    safe = np.where(a > 0, a, 1.0)
    _, p = np.frexp(safe)                    # safe = m * 2**p, 0.5 <= m < 1
    e = (p - 9).astype(np.int64)             # 448 ~ 2**8.8: estimate
    for _ in range(4):                       # corrections are at most a step
        up = a > 448.0 * np.ldexp(1.0, e)
        e = np.where(up, e + 1, e)
        down = a <= 448.0 * np.ldexp(1.0, e - 1)
        e = np.where(down & (a > 0), e - 1, e)
    e = np.where(a > 0, e, -127)
    return np.clip(e, -127, 127)
