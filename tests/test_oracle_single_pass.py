"""Pins for the oracle's single-pass FC2 with online amax compensation
("miniTE technical report", section 5.6), CPU only.

The compensation has a closed form: after the last tile,
O * gs_last = sum_i gs_i * dO_i, so Y is the plain FC2 of the activation
whose tile i is dequantised against the scale gs_i it was encoded with.  The
tests check that form with an independent dequantise-then-multiply, the
running amax by brute force, the tile codes against the exact-real encoding,
the two cases where the single pass must reproduce the two-pass path (one
tile; every row's amax inside its first tile), all-zero rows and rows that
start with zero tiles, and the error band against the unquantised FC2.
"""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q
from oracle import moe as MO
from oracle import metrics as Mx
from microscaled_precision_moe_gb300 import synth


def _bf16(a):
    return F.bf16_round(np.asarray(a, dtype=np.float64)).astype(np.float32)


def _case(rows=(9, 0, 12), H=48, I=96, seed=0):
    """D [R, I] with a spread of row magnitudes, late outliers that raise the
    running amax, one all-zero row and one row whose first 48 columns are
    zero; W2 [E, H, I] quantised per expert.  Segments are unpadded."""
    rng = np.random.default_rng(seed)
    E = len(rows)
    seg = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    R = int(seg[-1])
    d = rng.standard_normal((R, I)) * np.exp(rng.standard_normal((R, 1)))
    late = rng.random((R, I)) < 0.03
    late[:, :I // 3] = False
    d = np.where(late, d * 20.0, d)
    d[0] = 0.0
    d[1, :48] = 0.0
    d = _bf16(d)
    w2 = _bf16(rng.standard_normal((E, H, I)) * 0.02)
    return d, seg, Q.nvfp4_quantize_joint([w2], E), w2


def _tiles(I, tile_k):
    return [(c0, min(c0 + tile_k, I)) for c0 in range(0, I, tile_k)]


def _dequant_by_tile(s, I, tile_k):
    """Each element decoded as q * s_b * gs_i, gs_i the scale of its tile."""
    gs_col = np.zeros(s["codes"].shape)
    for i, (c0, c1) in enumerate(_tiles(I, tile_k)):
        gs_col[:, c0:c1] = s["gs"][:, i:i + 1]
    sb = np.repeat(F.e4m3_decode(s["sb"]), Q.NV_BLOCK, axis=1)
    return F.e2m1_decode(s["codes"]) * sb * gs_col


def _two_pass_fc2(d, seg, w2q):
    qd, sd, tsd = Q.nvfp4_quantize_per_token(d)
    y = MO.grouped_gemm(Q.nvfp4_dequantize(qd, sd, tsd), MO.dequant_weights_nvfp4(w2q), seg)
    return qd, sd, tsd, y


@pytest.mark.parametrize("tile_k", [16, 32, 64, 96])
def test_compensation_closed_form(tile_k):
    """Y equals W2's full dequantisation applied to the tile-wise
    dequantised activation (64 gives a ragged 64 + 32 split of I = 96)."""
    d, seg, w2q, _ = _case()
    I = d.shape[1]
    s = MO.nvfp4_fc2_online_amax(d, seg, w2q, tile_k)
    xhat = _dequant_by_tile(s, I, tile_k)
    bw = MO.dequant_weights_nvfp4(w2q)
    ref = np.zeros_like(s["y64"])
    for e in range(len(seg) - 1):
        for r in range(int(seg[e]), int(seg[e + 1])):
            ref[r] = bw[e] @ xhat[r]
    tol = 1e-12 * np.max(np.abs(ref))
    assert np.max(np.abs(s["y64"] - ref)) <= tol
    assert np.array_equal(s["y"], F.bf16_round(s["y64"]))


def test_running_amax_brute_force():
    """gs of tile i is fl32(max of |D| over the row's columns [0, end of
    tile i]) / 2688), taken element by element; 0 while that max is 0."""
    d, seg, w2q, _ = _case()
    R, I = d.shape
    tile_k = 32
    s = MO.nvfp4_fc2_online_amax(d, seg, w2q, tile_k)
    for r in range(R):
        run = 0.0
        for i, (c0, c1) in enumerate(_tiles(I, tile_k)):
            for c in range(c0, c1):
                run = max(run, abs(float(d[r, c])))
            want = np.float32(run) / np.float32(2688.0) if run > 0 else np.float32(0.0)
            assert s["gs"][r, i] == want, (r, i)
    assert np.all(s["gs"][0] == 0) and np.all(s["codes"][0] == 0) and np.all(s["y"][0] == 0)
    assert np.all(s["gs"][1, :1] == 0) and s["gs"][1, 1] > 0      # zero first tile (48 cols)
    grew = np.diff(s["gs"], axis=1) > 0
    assert grew.any(), "the case must raise the running amax after the first tile"


def _near_midpoint(v, grid, rel=1e-6):
    """True where |v| lies within ``rel`` of the midpoint of two adjacent
    grid values (a rounding tie up to fp32 error)."""
    mids = (grid[1:] + grid[:-1]) / 2.0
    a = np.abs(np.asarray(v, dtype=np.float64))[..., None]
    return np.any(np.abs(a - mids) <= rel * mids, axis=-1)


def test_tile_codes_match_exact_real_encoding():
    """Each tile's block scales and codes are the NVFP4 encoding against that
    tile's gs.  The exact-real encoding (rational arithmetic) differs from the
    fp32 sequence only where the fp32 rounding of gs, 6 gs or the reciprocal
    moves a value across a rounding tie: every differing block scale has
    bmax / (6 gs) at an E4M3 midpoint, every differing code (in a block whose
    scale agrees) has x / (s_b gs) at an E2M1 midpoint, one step apart.  (With
    bf16 data such ties are not rare: here 22.5 and 8.4375 give exactly 168,
    half way between 160 and 176.)  No block scale saturates, because the
    running amax includes the tile being encoded."""
    d, seg, w2q, _ = _case()
    R, I = d.shape
    tile_k = 32
    s = MO.nvfp4_fc2_online_amax(d, seg, w2q, tile_k)
    e4_grid = F.E4M3_GRID[:0x7F]
    n_blocks = n_codes = 0
    for i, (c0, c1) in enumerate(_tiles(I, tile_k)):
        g = s["gs"][:, i].astype(np.float64)
        q, sb = Q.nvfp4_encode_exact(d[:, c0:c1], s["gs"][:, i])
        got_sb = s["sb"][:, c0 // 16:c1 // 16]
        blk = np.abs(d[:, c0:c1].astype(np.float64)).reshape(R, -1, 16).max(axis=2)
        bad_b = sb != got_sb
        for r, b in np.argwhere(bad_b):
            assert _near_midpoint(blk[r, b] / (6.0 * g[r]), e4_grid), (i, r, b)
            assert abs(int(sb[r, b]) - int(got_sb[r, b])) == 1, (i, r, b)
        n_blocks += int(bad_b.sum())
        got_q = s["codes"][:, c0:c1]
        ok_blk = np.repeat(~bad_b, 16, axis=1)
        for r, c in np.argwhere((q != got_q) & ok_blk):
            den = F.e4m3_decode(got_sb[r, c // 16]) * g[r]
            assert _near_midpoint(float(d[r, c0 + c]) / den, F.E2M1_GRID), (i, r, c)
            assert q[r, c] >> 3 == got_q[r, c] >> 3, (i, r, c)
            assert abs(int(q[r, c] & 7) - int(got_q[r, c] & 7)) == 1, (i, r, c)
            n_codes += 1
    assert n_blocks <= 2 and n_codes <= 4, (n_blocks, n_codes)
    live = s["gs"].max(axis=1) > 0
    assert np.all(F.e4m3_decode(s["sb"][live]) <= 448.0)
    # blocks holding the running amax are encoded with s_b * gs = amax / 6 up
    # to E4M3 rounding, so their largest code is 6 or its neighbour 4
    assert np.any(s["codes"] & 0x7 == 7)


@pytest.mark.parametrize("tile_k", [96, 256])
def test_one_tile_is_the_two_pass_path(tile_k):
    """A tile as wide as I: the running amax is the row amax, so codes,
    scales and Y are those of whole-row re-quantisation."""
    d, seg, w2q, _ = _case()
    s = MO.nvfp4_fc2_online_amax(d, seg, w2q, tile_k)
    qd, sd, tsd, y2 = _two_pass_fc2(d, seg, w2q)
    assert s["gs"].shape[1] == 1
    assert np.array_equal(s["gs"][:, 0], tsd)
    assert np.array_equal(s["codes"], Q.unpack_e2m1(qd))
    assert np.array_equal(s["sb"], sd)
    assert np.max(np.abs(s["y64"] - y2)) <= 1e-12 * np.max(np.abs(y2))


@pytest.mark.parametrize("tile_k", [16, 48])
def test_amax_in_first_tile_is_the_two_pass_path(tile_k):
    """When each row's amax sits in its first tile, gs never changes and the
    single pass reproduces the two-pass codes and Y for any tile width."""
    d, seg, w2q, _ = _case()
    d = d.copy()
    d[1, :48] = d[1, 48:96]                        # no leading zero tile here
    amax = np.max(np.abs(d), axis=1)
    d[:, 3] = np.where(amax > 0, -amax, 0.0).astype(np.float32)
    s = MO.nvfp4_fc2_online_amax(d, seg, w2q, tile_k)
    qd, sd, tsd, y2 = _two_pass_fc2(d, seg, w2q)
    assert np.all(s["gs"] == tsd[:, None])
    assert np.array_equal(s["codes"], Q.unpack_e2m1(qd))
    assert np.array_equal(s["sb"], sd)
    assert np.max(np.abs(s["y64"] - y2)) <= 1e-12 * np.max(np.abs(y2))


def test_layer_error_band_against_two_pass():
    """On a reduced 30B-A3B-shaped layer the single pass stays in the two-pass
    path's NVFP4 error band (relative Frobenius error of Y against the
    unquantised FC2 of the same D and W2 within 5 % of the two-pass error),
    tokens whose rows all keep their first-tile scale get the two-pass output
    bit for bit, and padding rows stay zero."""
    shape = synth.scaled(synth.MOE_30B, T=64, H=256, I=512, E=4, k=2)
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape).float().numpy()
    w1, w2 = (w.float().numpy() for w in synth.moe_weights(shape))
    with np.errstate(over="ignore"):
        s = MO.nvfp4_moe_forward_single_pass(x, ids.numpy(), prob.numpy(), w1, w2, shape.E,
                                             tile_k=128)
    r = s["two_pass"]
    exact = MO.grouped_gemm(r["d"].astype(np.float64), w2.astype(np.float64), r["seg"])
    y2 = MO.grouped_gemm(Q.nvfp4_dequantize(r["qd"], r["sd"], r["tsd"]),
                         MO.dequant_weights_nvfp4(r["w2"]), r["seg"])
    e1, e2 = Mx.rel_frobenius(s["y64"], exact), Mx.rel_frobenius(y2, exact)
    assert 0.05 < e2 < 0.3 and abs(e1 - e2) <= 0.05 * e2, (e1, e2)
    assert Mx.rel_frobenius(s["y64"], y2) < 0.1
    assert np.all(s["y"][r["perm"] < 0] == 0)
    same = np.all(s["gs"] == r["tsd"][:, None], axis=1)
    assert np.array_equal(s["y"][same], r["y"][same])
    inv = r["inv"].reshape(shape.T, shape.k)
    tok = same[inv].all(axis=1)
    assert tok.any() and np.array_equal(s["out"][tok], r["out"][tok])
