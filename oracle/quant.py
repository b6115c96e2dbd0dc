"""MXFP8 and NVFP4 quantisers, the scale-tile layout and dequantisation.

Oracle: test infrastructure only.

MXFP8 (1-D blocks of 32, one E8M0 power-of-two scale per block, rounded up
so the block max never clips; a row-wise 1x32 copy and a column-wise 32x1
copy, each quantised independently from the full-precision input):
"Towards Blackwell-native 8-bit and 4-bit RL", sections "Format background /
MXFP8" and "Recipe 1: end-to-end MXFP8 RL / Training".

NVFP4 (E2M1 codes, one E4M3 scale per 16 values rounded to nearest, an FP32
outer scale, decode x_hat = q * s_b * s_g): same post, section "Format
background / NVFP4"; "miniTE technical report", section 2.2.  The outer scale
is per token for activations (post, section "Per-token activation scaling";
report, sections 2.3 and 5.1) and shared by gate and up for a weight (post,
same section).  Its value is s_g = amax / 2688 = amax / (448 * 6) (report,
section 5.6).

Canonical fp32 sequence (every step IEEE binary32, round to nearest even,
no fused multiply-add, subnormals kept).  The pages fix the rules, not the
operation order; this order is the contract the CUDA kernels follow:

  1. a   = max_j |x_j|                       (or the caller's amax)
  2. s_g = fl(a / 2688);  if 0 < s_g < 2**-116: s_g = 2**-116;  a = 0 -> s_g = 0
  3. per block of 16:  s_b = E4M3( fl(bmax / fl(6 * s_g)) )
  4. s_b = 0 -> every code of the block is 0;  else r = fl(1 / fl(s_b * s_g)),
     q_j = E2M1( fl(x_j * r) )

The 2**-116 floor is a reading (the pages give none): it keeps every later
intermediate finite and normal for rows whose amax is below about 3e-32.

Packing: element 2j in the low nibble, 2j+1 in the high nibble.

Scale layout for the tensor cores (a reading; the pages do not print it): the
[rows, cols] scale matrix is padded to rows % 128 == 0 and cols % 4 == 0 with
zero bytes and cut into 128 x 4 tiles; tile (rt, ct) starts at byte
(rt * cols_pad / 4 + ct) * 512 and holds entry (r, c) at
(r % 32) * 16 + (r // 32) * 4 + c.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

NVFP4_OUTER_DIV = np.float32(2688.0)      # 448 * 6, report section 5.6
NVFP4_SG_FLOOR = np.float32(2.0 ** -116)  # reading: keeps intermediates normal
MX_BLOCK = 32
NV_BLOCK = 16


def pad_to(n: int, m: int) -> int:
    return (n + m - 1) // m * m


def scale_bytes(rows: int, cols: int) -> int:
    return pad_to(rows, 128) * pad_to(cols, 4)


# ------------------------------------------------------------ scale layout

def swizzle_scales(s: np.ndarray) -> np.ndarray:
    """Row-major [rows, cols] uint8 scales -> flat 128x4-tiled byte array."""
    rows, cols = s.shape
    rp, cp = pad_to(rows, 128), pad_to(cols, 4)
    out = np.zeros(rp * cp, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    rt, rr = r // 128, r % 128
    ct, cc = c // 4, c % 4
    off = (rt * (cp // 4) + ct) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc
    out[off] = s
    return out


def unswizzle_scales(flat: np.ndarray, rows: int, cols: int) -> np.ndarray:
    cp = pad_to(cols, 4)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    rt, rr = r // 128, r % 128
    ct, cc = c // 4, c % 4
    off = (rt * (cp // 4) + ct) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc
    return np.asarray(flat)[off]


# ------------------------------------------------------------ MXFP8

def mxfp8_quantize_blocks(v: np.ndarray):
    """Quantise blocks laid along the last axis (length 32 each).

    v: float array [..., nblk, 32] of bf16 values.  Returns (codes uint8 of
    the same shape, scale bytes uint8 [..., nblk]).
    1. a = max |v| over the block (exact);
    2. e = smallest integer with a <= 448 * 2**e, clamped to [-127, 127];
       scale byte = e + 127;
    3. code = E4M3(v * 2**-e)  (the product is exact in fp64).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.max(np.abs(v), axis=-1)
    e = F.e8m0_exponent_for_amax(a)
    scaled = v * np.ldexp(1.0, -e)[..., None]
    # the kernel forms this product in fp32; a value whose product is an fp32
    # subnormal lies below half the smallest E4M3 subnormal and encodes to 0
    # either way, so the fp64 product gives the same code
    codes = F.e4m3_encode(scaled)
    return codes, (e + 127).astype(np.uint8)


def mxfp8_quantize_rowwise(x: np.ndarray):
    """x [M, K] (K % 32 == 0) -> codes [M, K], scales [M, K/32] (row-major)."""
    M, K = x.shape
    assert K % MX_BLOCK == 0
    codes, s = mxfp8_quantize_blocks(x.reshape(M, K // MX_BLOCK, MX_BLOCK))
    return codes.reshape(M, K), s


def mxfp8_quantize_colwise(x: np.ndarray):
    """x [M, K] -> transposed codes [K, M], scales [K, ceil(M/32)].

    Column blocks are 32 consecutive rows of one column.  A partial last block
    behaves as if padded with zeros (its amax is that of the real rows).
    """
    M, K = x.shape
    Mp = pad_to(M, MX_BLOCK)
    xt = np.zeros((K, Mp), dtype=np.float64)
    xt[:, :M] = np.asarray(x, dtype=np.float64).T
    codes, s = mxfp8_quantize_blocks(xt.reshape(K, Mp // MX_BLOCK, MX_BLOCK))
    return codes.reshape(K, Mp)[:, :M].copy(), s


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes [R, C] with row-major scales [R, ceil(C/32)] -> fp64 values."""
    R, C = codes.shape
    s = F.e8m0_decode(scales)
    rep = np.repeat(s, MX_BLOCK, axis=1)[:, :C]
    return F.e4m3_decode(codes) * rep


# ------------------------------------------------------------ NVFP4

def nvfp4_outer_scale(a: np.ndarray) -> np.ndarray:
    """Step 2: s_g = fl(a / 2688) with the 2**-116 floor; 0 for a = 0."""
    a = np.asarray(a, dtype=np.float32)
    sg = (a / NVFP4_OUTER_DIV).astype(np.float32)
    sg = np.where((a > 0) & (sg < NVFP4_SG_FLOOR), NVFP4_SG_FLOOR, sg)
    return np.where(a > 0, sg, np.float32(0.0)).astype(np.float32)


def nvfp4_encode_with_outer(x: np.ndarray, sg: np.ndarray):
    """Steps 3-4 for rows that share an outer scale.

    x: float32 [R, K] (bf16 values), sg: float32 [R] (0 for an all-zero row).
    Returns (codes uint8 [R, K] in 0..15, block scale bytes [R, K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    R, K = x.shape
    assert K % NV_BLOCK == 0
    xb = x.reshape(R, K // NV_BLOCK, NV_BLOCK)
    bmax = np.max(np.abs(xb), axis=-1).astype(np.float32)          # exact
    sg2 = np.asarray(sg, dtype=np.float32)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        six_sg = (np.float32(6.0) * sg2).astype(np.float32)
        sbf = (bmax / six_sg).astype(np.float32)
    sbf = np.where(sg2 > 0, sbf, np.float32(0.0))
    sb_code = F.e4m3_encode(sbf)                                  # RNE, satfinite
    sb = F.e4m3_decode(sb_code).astype(np.float32)                # exact in fp32
    with np.errstate(divide="ignore", over="ignore"):
        prod = (sb * sg2).astype(np.float32)
        r = (np.float32(1.0) / prod).astype(np.float32)
    r = np.where(sb > 0, r, np.float32(0.0))
    y = (xb * r[..., None]).astype(np.float32)
    q = F.e2m1_encode(y)
    q = np.where((sb > 0)[..., None], q, np.uint8(0))
    return q.reshape(R, K).astype(np.uint8), sb_code.astype(np.uint8)


def nvfp4_quantize_per_token(x: np.ndarray, amax=None):
    """Per-token NVFP4.  x [M, K] bf16 values (any float dtype holding them).

    ``amax`` (optional, [M] float32) replaces step 1 with the producer's row
    amax (report section 5.3); with the true row maximum the result is the
    same.  Returns (packed uint8 [M, K/2], block scales uint8 [M, K/16]
    row-major, s_g float32 [M]).
    """
    x = np.asarray(x, dtype=np.float32)
    if amax is None:
        a = np.max(np.abs(x), axis=1).astype(np.float32)
    else:
        a = np.asarray(amax, dtype=np.float32)
    sg = nvfp4_outer_scale(a)
    q, sb = nvfp4_encode_with_outer(x, sg)
    return pack_e2m1(q), sb, sg


def nvfp4_quantize_joint(parts, E: int):
    """Joint-scale weight quantisation (gate and up share s_g).

    parts: list of arrays [E, rows_p, K]; per expert e the outer scale comes
    from the amax over all parts' rows of that expert, and the quantised rows
    are the parts concatenated in order.  Returns (packed [E, R, K/2],
    block scales [E, R, K/16], s_g float32 [E]).
    """
    cat = np.concatenate([np.asarray(p, dtype=np.float32) for p in parts], axis=1)
    E_, R, K = cat.shape
    assert E_ == E
    a = np.max(np.abs(cat.reshape(E, -1)), axis=1).astype(np.float32)
    sg = nvfp4_outer_scale(a)
    q, sb = nvfp4_encode_with_outer(cat.reshape(E * R, K), np.repeat(sg, R))
    return pack_e2m1(q).reshape(E, R, K // 2), sb.reshape(E, R, K // NV_BLOCK), sg


def pack_e2m1(q: np.ndarray) -> np.ndarray:
    q = np.asarray(q, dtype=np.uint8)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(p: np.ndarray) -> np.ndarray:
    p = np.asarray(p, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def nvfp4_dequantize(packed: np.ndarray, sb: np.ndarray, sg) -> np.ndarray:
    """x_hat = q * s_b * s_g in fp64 (exact).  packed [R, K/2], sb [R, K/16],
    sg scalar or [R]."""
    q = F.e2m1_decode(unpack_e2m1(packed))
    s = np.repeat(F.e4m3_decode(sb), NV_BLOCK, axis=-1)
    sg = np.asarray(sg, dtype=np.float64)
    if sg.ndim == 1:
        sg = sg[:, None]
    return q * s * sg


def nvfp4_dequantize_bf16(packed: np.ndarray, sb: np.ndarray, sg) -> np.ndarray:
    """The BF16 dequantisation the dequantized backward feeds to its BF16
    GEMMs ("Towards Blackwell-native 8-bit and 4-bit RL", section
    "High-precision and dequantized backward"): the exact value q * s_b * s_g
    rounded once to the nearest bf16 (ties to even).  Returned as fp64."""
    return F.bf16_round(nvfp4_dequantize(packed, sb, sg))


def mxfp8_dequantize_bf16(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP8 counterpart (same section): q * 2^e rounded once to bf16 (exact
    unless the value falls below bf16's normal range)."""
    return F.bf16_round(mxfp8_dequantize(codes, scales))


def nvfp4_encode_exact(x: np.ndarray, sg: np.ndarray):
    """The same encoding with each rounding taken once on the exact real value.

    s_b = E4M3(bmax / (6 s_g)) and q = E2M1(x / (s_b s_g)), computed in
    rational arithmetic (python Fractions) instead of the fp32 sequence.  Used
    to report how often the fp32 reciprocal-multiply order departs from the
    exact-real encoding.  Slow: small inputs only.
    """
    from fractions import Fraction
    x = np.asarray(x, dtype=np.float32)
    R, K = x.shape
    sbc = np.zeros((R, K // NV_BLOCK), dtype=np.uint8)
    q = np.zeros((R, K), dtype=np.uint8)
    e4 = [Fraction(float(v)) for v in F.E4M3_GRID]
    e2 = [Fraction(float(v)) for v in F.E2M1_GRID]

    def nearest(v: Fraction, grid, ties_even=True):
        best, bi = None, 0
        for i, g in enumerate(grid):
            d = abs(v - g)
            if best is None or d < best or (d == best and i % 2 == 0):
                best, bi = d, i
        return bi

    for r in range(R):
        s = Fraction(float(sg[r]))
        if s == 0:
            continue
        for b in range(K // NV_BLOCK):
            blk = x[r, b * NV_BLOCK:(b + 1) * NV_BLOCK]
            bmax = Fraction(float(np.max(np.abs(blk))))
            sb = nearest(bmax / (6 * s), e4)
            sbc[r, b] = sb
            if sb == 0:
                continue
            den = e4[sb] * s
            for j, v in enumerate(blk):
                fv = Fraction(float(v))
                c = nearest(abs(fv) / den, e2)
                if fv < 0 or (fv == 0 and np.signbit(v)):
                    c |= 0x8
                q[r, b * NV_BLOCK + j] = c
    return q, sbc
