"""Pins for the oracle's MXFP8 / NVFP4 quantisers (CPU only).

What fixes each expectation is outside the quantiser code: exactly
representable round trips, closed forms, the all-zero / max / subnormal
extremes, batch independence, an exact-rational re-encoding, an independent
construction of the scale-tile layout, and the storage sizes printed in the
memory tables of "Towards Blackwell-native 8-bit and 4-bit RL" (section
"Backward cost and memory").
"""
import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q
from oracle import metrics as Mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    return F.bf16_round(np.asarray(a, dtype=np.float64)).astype(np.float32)


# ------------------------------------------------------------------ MXFP8

@pytest.mark.parametrize("k", [-20, -3, 0, 5, 30])
def test_mxfp8_roundtrip_exact(k):
    """A block whose max is 448 * 2**k and whose other elements are E4M3 grid
    values times 2**k encodes exactly with scale byte 127 + k."""
    rng = np.random.default_rng(k + 100)
    codes = rng.integers(0, 0x7F, size=(4, 32))
    codes[:, 5] = 0x7E                                   # block max = 448
    sign = rng.integers(0, 2, size=(4, 32)) * 0x80
    vals = F.e4m3_decode(codes | sign) * 2.0 ** k
    x = vals.astype(np.float32)
    assert np.array_equal(_bf16(x), x)                   # bf16-representable
    q, s = Q.mxfp8_quantize_rowwise(x)
    assert np.all(s == 127 + k)
    assert np.array_equal(Q.mxfp8_dequantize(q, s), vals)
    assert np.array_equal(q, (codes | sign).astype(np.uint8))


def test_mxfp8_colwise_is_rowwise_of_transpose():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((96, 64)) * np.exp(rng.standard_normal((96, 1)) * 3))
    qc, sc = Q.mxfp8_quantize_colwise(x)
    qr, sr = Q.mxfp8_quantize_rowwise(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr) and np.array_equal(sc, sr)


def test_mxfp8_colwise_partial_block_is_zero_padded():
    rng = np.random.default_rng(4)
    x = _bf16(rng.standard_normal((40, 32)))
    qc, sc = Q.mxfp8_quantize_colwise(x)
    assert qc.shape == (32, 40) and sc.shape == (32, 2)
    xp = np.zeros((64, 32), dtype=np.float32)
    xp[:40] = x
    qp, sp = Q.mxfp8_quantize_colwise(xp)
    assert np.array_equal(qp[:, :40], qc) and np.array_equal(sp, sc)


def test_mxfp8_extremes():
    K = 64
    zeros = np.zeros((2, K), dtype=np.float32)
    q, s = Q.mxfp8_quantize_rowwise(zeros)
    assert np.all(q == 0) and np.all(s == 0)
    maxes = np.where(np.arange(2 * K).reshape(2, K) % 3 == 0, -448.0, 448.0).astype(np.float32)
    q, s = Q.mxfp8_quantize_rowwise(maxes)
    assert np.all(s == 127) and np.all((q & 0x7F) == 0x7E)
    assert not np.any(q == 0xFF) and not np.any(s == 0xFF)
    # bf16 subnormals: the scale clamps at 2**-127 (byte 0x00)
    sub = F.bf16_bits_to_f32(np.arange(1, 1 + 2 * K, dtype=np.uint16) % 127 + 1).reshape(2, K)
    q, s = Q.mxfp8_quantize_rowwise(sub)
    assert np.all(s == 0)
    # the codes are the E4M3 encodings of v * 2**127 (exact product)
    assert np.array_equal(q, F.e4m3_encode(sub.astype(np.float64) * 2.0 ** 127))
    # huge values: bf16 max never produces NaN or 0xFF
    big = np.full((1, 32), F.bf16_bits_to_f32(np.array([0x7F7F], np.uint16))[0])
    q, s = Q.mxfp8_quantize_rowwise(big.astype(np.float32))
    # a = 1.9921875 * 2**127: e = 120, scaled max 255 -> E4M3 256 (code 0x78)
    assert s[0, 0] == 127 + 120 and np.all(q == 0x78)


def test_mxfp8_error_bound():
    """Every element is within half an E4M3 step of its scaled value."""
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((64, 256)) * 10)
    q, s = Q.mxfp8_quantize_rowwise(x)
    xh = Q.mxfp8_dequantize(q, s)
    scale = np.repeat(F.e8m0_decode(s), 32, axis=1)
    # E4M3 relative spacing <= 2**-3 for normal codes, absolute 2**-9 below
    err = np.abs(xh - x) / scale
    bound = np.maximum(np.abs(x) / scale * 2.0 ** -4, 2.0 ** -10)
    assert np.all(err <= bound + 1e-300)


# ------------------------------------------------------------------ NVFP4

@pytest.mark.parametrize("k", [-40, -10, 0, 7, 60])
def test_nvfp4_roundtrip_exact(k):
    """A row with amax 2688 * 2**k has s_g = 2**k; a block whose max is the row
    amax gets s_b = 448; elements q * 448 * 2**k encode exactly."""
    rng = np.random.default_rng(k + 100)
    K = 64
    q = rng.integers(0, 16, size=(3, K)).astype(np.uint8)
    q[:, ::16] = 0x7                                     # each block max = 6
    vals = F.e2m1_decode(q) * 448.0 * 2.0 ** k
    x = vals.astype(np.float32)
    assert np.array_equal(_bf16(x), x)
    packed, sb, sg = Q.nvfp4_quantize_per_token(x)
    assert np.all(sg == np.float32(2.0 ** k))
    assert np.all(F.e4m3_decode(sb) == 448.0)
    assert np.array_equal(Q.unpack_e2m1(packed) & 0x7, q & 0x7)
    assert np.array_equal(Q.nvfp4_dequantize(packed, sb, sg), vals)


def test_nvfp4_outer_scale_is_amax_over_2688():
    # report section 5.6: gs = gamax / 2688
    a = np.array([2688.0, 1.0, 448.0 * 6 * 3, 1e-3], dtype=np.float32)
    sg = Q.nvfp4_outer_scale(a)
    assert sg[0] == 1.0 and sg[2] == 3.0
    assert sg[1] == np.float32(1.0) / np.float32(2688.0)
    assert sg[3] == np.float32(np.float32(1e-3) / np.float32(2688.0))


def test_nvfp4_extremes():
    K = 32
    packed, sb, sg = Q.nvfp4_quantize_per_token(np.zeros((2, K), np.float32))
    assert np.all(packed == 0) and np.all(sb == 0) and np.all(sg == 0)
    bmax = F.bf16_bits_to_f32(np.array([0x7F7F], np.uint16))[0]
    x = np.full((2, K), bmax, dtype=np.float32)
    x[1, ::2] *= -1
    packed, sb, sg = Q.nvfp4_quantize_per_token(x)
    assert np.all(np.isfinite(sg)) and np.all(sb == 0x7E)
    q = Q.unpack_e2m1(packed)
    assert np.all((q & 0x7) == 0x7)
    assert np.all(np.isfinite(Q.nvfp4_dequantize(packed, sb, sg)))
    # a row of bf16 subnormals: the 2**-116 floor keeps everything finite
    sub = F.bf16_bits_to_f32(np.arange(1, 1 + K, dtype=np.uint16)).reshape(1, K)
    packed, sb, sg = Q.nvfp4_quantize_per_token(sub)
    assert sg[0] == np.float32(2.0 ** -116)
    assert np.all(np.isfinite(Q.nvfp4_dequantize(packed, sb, sg)))
    # a single nonzero element in an otherwise zero row
    one = np.zeros((1, K), np.float32)
    one[0, 17] = -3.0
    packed, sb, sg = Q.nvfp4_quantize_per_token(one)
    xh = Q.nvfp4_dequantize(packed, sb, sg)
    assert sb[0, 0] == 0 and F.e4m3_decode(sb[0, 1]) == 448.0
    assert abs(xh[0, 17] + 3.0) <= 3.0 * 2 ** -8 and np.count_nonzero(xh) == 1


def test_nvfp4_amax_reuse_matches_own_amax():
    rng = np.random.default_rng(9)
    x = _bf16(rng.standard_normal((16, 128)) * 5)
    a = np.max(np.abs(x), axis=1).astype(np.float32)
    r1 = Q.nvfp4_quantize_per_token(x)
    r2 = Q.nvfp4_quantize_per_token(x, amax=a)
    for u, v in zip(r1, r2):
        assert np.array_equal(u, v)


def test_nvfp4_batch_independence():
    """A token's bytes do not depend on the batch it is quantised in
    (post, section "Per-token activation scaling")."""
    rng = np.random.default_rng(11)
    x = _bf16(rng.standard_normal((64, 256)) * np.exp(rng.standard_normal((64, 1)) * 4))
    full = Q.nvfp4_quantize_per_token(x)
    perm = rng.permutation(64)
    permuted = Q.nvfp4_quantize_per_token(x[perm])
    for t in [0, 13, 63]:
        alone = Q.nvfp4_quantize_per_token(x[t:t + 1])
        assert np.array_equal(alone[0][0], full[0][t])
        assert np.array_equal(alone[1][0], full[1][t])
        assert alone[2][0] == full[2][t]
    for u, v in zip(full, permuted):
        assert np.array_equal(u[perm], v)


def test_mxfp8_batch_independence_rows():
    rng = np.random.default_rng(12)
    x = _bf16(rng.standard_normal((64, 128)))
    q, s = Q.mxfp8_quantize_rowwise(x)
    q1, s1 = Q.mxfp8_quantize_rowwise(x[5:6])
    assert np.array_equal(q1[0], q[5]) and np.array_equal(s1[0], s[5])


def test_nvfp4_joint_scale_shared_by_gate_and_up():
    rng = np.random.default_rng(13)
    g = _bf16(rng.standard_normal((2, 8, 64)) * 0.02)
    u = _bf16(rng.standard_normal((2, 8, 64)) * 0.02)
    u[1, 3, 7] = 5.0                                      # outlier in up of expert 1
    packed, sb, sg = Q.nvfp4_quantize_joint([g, u], 2)
    a = np.max(np.abs(np.concatenate([g, u], axis=1).reshape(2, -1)), axis=1)
    assert np.array_equal(sg, Q.nvfp4_outer_scale(a.astype(np.float32)))
    assert sg[1] == np.float32(np.float32(5.0) / np.float32(2688.0))
    # gate rows of expert 1 are quantised with the outer scale set by up
    pg, sbg, _ = Q.nvfp4_quantize_joint([g], 2)
    assert not np.array_equal(pg[1], packed[1, :8]) or not np.array_equal(sbg[1], sb[1, :8])
    # each row equals the per-row encoding with the shared scale
    q, s = Q.nvfp4_encode_with_outer(np.concatenate([g[1], u[1]]), np.full(16, sg[1]))
    assert np.array_equal(Q.pack_e2m1(q), packed[1]) and np.array_equal(s, sb[1])


def test_nvfp4_fp32_order_vs_exact_real_encoding():
    """The fp32 reciprocal-multiply sequence departs from the exact-real
    encoding at most rarely, and then by one code step."""
    rng = np.random.default_rng(21)
    x = _bf16(rng.standard_normal((24, 256)) * np.exp(rng.standard_normal((24, 1)) * 2))
    x[0, :16] = 0
    sg = Q.nvfp4_outer_scale(np.max(np.abs(x), axis=1))
    q, sb = Q.nvfp4_encode_with_outer(x, sg)
    qe, sbe = Q.nvfp4_encode_exact(x, sg)
    assert np.array_equal(sb, sbe)
    diff = q != qe
    assert diff.mean() <= 1e-3
    if diff.any():
        dv = np.abs(F.e2m1_decode(q[diff]) - F.e2m1_decode(qe[diff]))
        assert np.all(dv <= 2.0)


def test_nvfp4_error_in_expected_band():
    """E2M1 with E4M3 block scales on Gaussian data: relative L2 near 0.1
    (the report's E2M1 figure on real inputs is 0.1014, section 2.3)."""
    rng = np.random.default_rng(22)
    x = _bf16(rng.standard_normal((64, 1024)))
    packed, sb, sg = Q.nvfp4_quantize_per_token(x)
    r = Mx.rel_l2(Q.nvfp4_dequantize(packed, sb, sg), x)
    assert 0.05 < r < 0.13


# ------------------------------------------------------------------ layout

def test_scale_swizzle_layout():
    """Independent construction: walk 128x4 tiles in order; inside a tile the
    512 bytes are 32 lines of 16 bytes, line i holding rows i, i+32, i+64,
    i+96 (4 bytes each)."""
    rows, cols = 300, 10
    rng = np.random.default_rng(2)
    s = rng.integers(1, 255, size=(rows, cols)).astype(np.uint8)
    flat = Q.swizzle_scales(s)
    rp, cp = 384, 12
    assert flat.size == rp * cp == Q.scale_bytes(rows, cols)
    out = []
    for rt in range(rp // 128):
        for ct in range(cp // 4):
            for line in range(32):
                for j in range(4):
                    r = rt * 128 + j * 32 + line
                    for c in range(ct * 4, ct * 4 + 4):
                        out.append(s[r, c] if (r < rows and c < cols) else 0)
    assert np.array_equal(flat, np.array(out, dtype=np.uint8))
    assert np.array_equal(Q.unswizzle_scales(flat, rows, cols), s)


def test_storage_sizes_match_memory_tables():
    """Post, section "Backward cost and memory": the high-precision backward
    saves the column-wise copy of X (2048 x 2048) and W (8192 x 2048):
    -20.62 MB for MXFP8 and -11.25 MB for NVFP4 (MiB in the tables)."""
    gold = dict(l.split("=") for l in open(os.path.join(GOLDEN, "memory_tables.txt"))
                .read().split("\n") if l and not l.startswith("#"))
    total = 0
    for shape in [(2048, 2048), (8192, 2048)]:
        x = np.zeros(shape, np.float32)
        q, s = Q.mxfp8_quantize_colwise(x)
        total += q.nbytes + s.nbytes
    assert round(total / 2 ** 20, 2) == float(gold["mxfp8_colwise_mib"])
    total = 0
    for shape in [(2048, 2048), (8192, 2048)]:
        x = np.zeros(shape, np.float32)
        p, sb, sg = Q.nvfp4_quantize_per_token(np.ascontiguousarray(x.T))
        total += p.nbytes + sb.nbytes
    assert round(total / 2 ** 20, 2) == float(gold["nvfp4_second_copy_mib"])


# ------------------------------------------------------------------ dequantisation to bf16

def _bf16_grid_fractions():
    """Every non-negative finite bf16 value as an exact Fraction, ascending,
    with its bit pattern (brute-force rounding target)."""
    from fractions import Fraction
    bits = np.arange(0, 0x7F80, dtype=np.uint16)            # +0 .. largest finite
    vals = F.bf16_bits_to_f32(bits).astype(np.float64)
    return [Fraction(float(v)) for v in vals], bits


def _nearest_bf16_brute(v, grid, bits):
    """Round the exact rational v to the nearest bf16, ties to the even bit
    pattern, by search over every bf16 value."""
    import bisect
    mag = abs(v)
    i = bisect.bisect_left(grid, mag)
    if i < len(grid) and grid[i] == mag:
        j = i
    elif i == 0:
        j = 0
    else:
        lo, hi = i - 1, min(i, len(grid) - 1)
        dlo, dhi = mag - grid[lo], grid[hi] - mag
        j = lo if (dlo < dhi or (dlo == dhi and bits[lo] % 2 == 0)) else hi
    return float(grid[j]) * (-1.0 if v < 0 else 1.0)


def test_nvfp4_dequantize_bf16_brute_force():
    """q * s_b * s_g rounded once to bf16, against exact rational products and
    a search over all bf16 values; outer scales chosen to hit exact ties
    (1 + 2^-8 sits halfway between bf16 neighbours), plain inexact values and
    the bf16 subnormal range."""
    from fractions import Fraction
    grid, bits = _bf16_grid_fractions()
    rng = np.random.default_rng(5)
    K = 32
    sgs = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, np.float32(1.0 / 3.0), 2.0 ** -130,
                    np.float32(3.3e-39), np.float32(0.7071)], dtype=np.float32)
    R = len(sgs)
    q = rng.integers(0, 16, size=(R, K)).astype(np.uint8)
    sb = rng.integers(0, 0x7F, size=(R, K // 16)).astype(np.uint8)
    sb[:, 0] = 0x38                                          # s_b = 1
    packed = Q.pack_e2m1(q)
    got = Q.nvfp4_dequantize_bf16(packed, sb, sgs)
    qv, sv = F.e2m1_decode(q), F.e4m3_decode(sb)
    for r in range(R):
        for c in range(K):
            exact = Fraction(float(qv[r, c])) * Fraction(float(sv[r, c // 16])) * Fraction(float(sgs[r]))
            assert got[r, c] == _nearest_bf16_brute(exact, grid, bits), (r, c)
    # the tie row rounds to even: 1 * 1 * (1 + 2^-8) -> 1.0
    one = Q.pack_e2m1(np.array([[2] + [0] * 15], np.uint8))
    assert Q.nvfp4_dequantize_bf16(one, np.array([[0x38]], np.uint8),
                                   np.array([1.0 + 2.0 ** -8], np.float32))[0, 0] == 1.0
    # double-rounding trap: 1.5 * (1 + 109227 * 2^-23) rounds in fp32 onto a
    # bf16 tie (and from there down to 1.515625); the single rounding of the
    # exact product goes up
    trap = np.float32(1.0 + 109227 * 2.0 ** -23)
    onefive = Q.pack_e2m1(np.array([[3] + [0] * 15], np.uint8))
    v = Q.nvfp4_dequantize_bf16(onefive, np.array([[0x38]], np.uint8), np.array([trap]))[0, 0]
    assert v == 1.5234375
    assert F.bf16_round(np.array([float(np.float32(1.5 * float(trap)))]))[0] == 1.515625


def test_mxfp8_dequantize_bf16_exact_and_extreme():
    """E4M3 x 2^e is a bf16 value unless it drops below 2^-126 (then one
    rounding, checked by brute force)."""
    from fractions import Fraction
    grid, bits = _bf16_grid_fractions()
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 256, size=(3, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10                     # no NaN codes
    scales = np.array([[127, 140], [0, 3], [120, 1]], dtype=np.uint8)
    got = Q.mxfp8_dequantize_bf16(codes, scales)
    ev = F.e4m3_decode(codes)
    for r in range(3):
        for c in range(64):
            exact = Fraction(float(ev[r, c])) * Fraction(2) ** (int(scales[r, c // 32]) - 127)
            assert got[r, c] == _nearest_bf16_brute(exact, grid, bits), (r, c)
    normal = scales[:, :, None].repeat(32, axis=2).reshape(3, 64) >= 127
    assert np.array_equal(got[normal], Q.mxfp8_dequantize(codes, scales)[normal])
