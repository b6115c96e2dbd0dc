"""GPU parity of the tcgen05 block-scaled grouped GEMMs against the oracle's
fp64 GEMMs on the dequantised codes.  Tolerance (the contract of the path):
relative Frobenius error <= 1e-3 and max |err| <= 1e-2 * max |ref|, against
the oracle result rounded to the kernel's output dtype."""
import numpy as np
import pytest
import torch

from oracle import quant as Q
from oracle import moe as MO
from oracle import formats as F
from oracle import metrics as Mx
from microscaled_precision_moe_gb300 import synth
from tests.gpu_util import need_gpu, np_bf16, u8

pytestmark = pytest.mark.gpu

REL, ELEM = 1e-3, 1e-2
# Bounds of the chained NVFP4 comparison (FC1 -> re-quantise -> FC2 ->
# combine); the re-quantisation is discontinuous, so rows of D that the fp32
# tensor-core accumulation rounds to a neighbouring bf16 value get other FP4
# operands than the oracle's.  Measured on GB300 over the reduced layers of
# this file (the values each test prints): at most 3.8e-5 of D elements and
# 0.4 % of D rows differ, those rows' Y is within 2.0e-2 of the oracle's and
# the layer output within 1.5e-3.  The bounds keep a margin of about 2.5-5x.
D_ELEM_DIFF = 2e-4       # fraction of D elements that differ (each by one bf16 step at most)
D_ROW_DIFF = 0.02        # fraction of D rows with any differing element
REQUANT_REL = 0.05       # relative error of Y on those rows (NVFP4 re-quantisation noise)
LAYER_REL = 5e-3         # relative Frobenius error of the layer output


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _ops():
    from microscaled_precision_moe_gb300 import ops
    return ops


def _L():
    from microscaled_precision_moe_gb300 import _lib
    return _lib


def _pad(tile_m):
    """Segment padding a GEMM tile mode needs (the small-M kernel: 128 rows)."""
    return 128 if tile_m == 1 else tile_m


def _assert_close(got, ref, what):
    ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, REL, ELEM)
    assert ok, f"{what}: rel_frob={rf:.3e} max_err={mx:.3e} bound={bound:.3e}"


@pytest.mark.parametrize("tile_m", [128, 256, 1])
def test_nvfp4_single_expert_gate_up(tile_m):
    """128 x 2048 activations (0.1% x50 outliers) against jointly quantised
    768 x 2048 gate and up weights -> 128 x 1536 fp32 (one CTA per tile, or a
    CTA pair whose second half lies past the 128 rows)."""
    ops, L = _ops(), _L()
    x, wg, wu = synth.single_expert_inputs(device="cuda")
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    qw, sw, tsw = ops.nvfp4_quantize_weight([wg[None].contiguous(), wu[None].contiguous()])
    out = torch.empty(128, 1536, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_F32, 1, 128, 1536, 2048, None,
                         qx, qw[0], sx, 128, sw, 128, out, alpha_a=tsx, alpha_b=tsw, tile_m=tile_m)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    ref = MO.nvfp4_gemm_single(np_bf16(x), np_bf16(wg), np_bf16(wu))["c"]
    _assert_close(out.cpu().numpy(), ref.astype(np.float32), "single-expert NVFP4")


@pytest.mark.parametrize("kind,epi,M,N,K", [
    ("nvfp4", "bf16", 128, 1536, 2048),     # the single-expert shape, bf16 out
    ("nvfp4", "f32", 40, 256, 768),         # 3 k-blocks over a 2-CTA cluster (uneven split)
    ("nvfp4", "f32", 1, 512, 4096),         # one row, 16 k-blocks over 8 CTAs
    ("mxfp8", "f32", 100, 512, 1024),       # 8 k-blocks of 128
    ("mxfp8", "bf16", 128, 256, 256),       # 2 k-blocks
])
def test_single_group_split_k(kind, epi, M, N, K):
    """One dense group of at most 128 rows on the small-M path runs split K
    (a cluster of CTAs per 128 weight rows, fixed-order reduction of their
    fp32 partials): against the oracle's fp64 GEMM on the dequantised codes,
    and deterministic from call to call."""
    ops, L = _ops(), _L()
    x = synth.normal_bf16(5, 1, (M, K), "cuda", outlier_p=1e-3, outlier_mul=50.0)
    w = synth.normal_bf16(5, 2, (N, K), "cuda", std=0.02)
    dt = torch.float32 if epi == "f32" else torch.bfloat16
    e = L.EPI_F32 if epi == "f32" else L.EPI_BF16
    out = torch.empty(M, N, dtype=dt, device="cuda")
    xn, wn = np_bf16(x), np_bf16(w)
    if kind == "nvfp4":
        qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
        qw, sw, tsw = ops.nvfp4_quantize_weight([w[None].contiguous()])
        run = lambda o: ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, e, 1, M, N, K, None, qx, qw[0],
                                             sx, K // 16, sw, K // 16, o, alpha_a=tsx, alpha_b=tsw,
                                             tile_m=L.TILE_SMALL_M)
        rq, rs, rts = Q.nvfp4_quantize_per_token(xn)
        wp, ws, wg = Q.nvfp4_quantize_joint([wn[None]], 1)
        ref = Q.nvfp4_dequantize(rq, rs, rts) @ Q.nvfp4_dequantize(wp[0], ws[0], wg[0]).T
    else:
        mx = ops.mxfp8_quantize(x, colwise=False)
        wq = ops.mxfp8_quantize(w, colwise=False)
        run = lambda o: ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, e, 1, M, N, K, None,
                                             mx["row_q"], wq["row_q"], mx["row_s"], K // 32,
                                             wq["row_s"], K // 32, o, tile_m=L.TILE_SMALL_M)
        ref = MO.mx_rows(xn) @ MO.mx_rows(wn).T
    run(out)
    out2 = torch.empty_like(out)
    run(out2)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    assert torch.equal(out, out2), "split-K reduction is deterministic"
    got = out.cpu().float().numpy()
    _assert_close(got, ref.astype(np.float32) if epi == "f32" else F.bf16_round(ref),
                  f"split-K {kind} {M}x{N}x{K}")


def _grouped_nvfp4_setup(shape, seed=0, pad=128):
    ops = _ops()
    ids, prob = synth.routing(shape, seed)
    x = synth.moe_activations(shape, seed, device="cuda")
    w1, w2 = synth.moe_weights(shape, seed, device="cuda")
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), shape.E, pad=pad)
    return ids, prob, x, w1, w2, seg, perm, inv, rp, cap


def _chained_compare(d_gpu, y_gpu, out_gpu, r, k, what):
    """Compare a chained FC1 -> re-quantise -> FC2 -> combine result.

    The FP4 re-quantisation of D is discontinuous: where the kernel's fp32
    accumulation rounds an element of D to a neighbouring bf16 value (the
    oracle accumulates exactly in fp64), the row's codes or its amax, and so
    its outer scale, can change.  So: D itself meets the GEMM tolerance and
    differs from the oracle's D by at most one bf16 step per element in a
    small fraction of elements; rows of D that are bit-identical give
    bit-identical FP4 operands (the quantiser is byte-exact), so their Y rows
    and the outputs of tokens whose rows all match must meet the GEMM
    tolerance; every row stays within the NVFP4 re-quantisation noise.  Y is
    compared on routed rows: the small-M FC2 leaves a segment's padding rows
    unwritten (the combine never reads them)."""
    R = int(r["seg"][-1])
    d = d_gpu[:R]
    _assert_close(d, r["d"], f"{what}: FC1 SwiGLU D")
    diff = d != r["d"]
    # one bf16 step of the reference, or an absolute floor for values that
    # come out of cancellation in the K-long accumulation
    ulp = np.abs(r["d"]) * 2.0 ** -7
    floor = 1e-4 * np.max(np.abs(r["d"]))
    assert np.all(np.abs(d - r["d"]) <= np.maximum(ulp, floor)), f"{what}: D beyond one step"
    same = ~diff.any(axis=1)
    real = np.asarray(r["perm"])[:R] >= 0
    y = y_gpu[:R]
    rel_re = 0.0
    if (~same & real).any():
        m = ~same & real
        rel_re = float(np.linalg.norm(y[m] - r["y"][m]) / np.linalg.norm(r["y"][m]))
    rel_out = Mx.rel_frobenius(out_gpu, r["out"])
    print(f"PARITY-STATS {what}: D elements differing {diff.mean():.3e}, D rows differing "
          f"{1.0 - same.mean():.4f}, re-quantised rows rel {rel_re:.3e}, layer rel {rel_out:.3e}")
    assert diff.mean() < D_ELEM_DIFF, f"{what}: {diff.mean():.2e} of D elements differ"
    assert 1.0 - same.mean() < D_ROW_DIFF, f"{what}: {1.0 - same.mean():.3f} of D rows differ"
    _assert_close(y[same & real], r["y"][same & real], f"{what}: FC2 rows with identical operands")
    assert rel_re < REQUANT_REL, f"{what}: re-quantised rows differ by {rel_re:.3e}"
    rows_ok = np.ones(R, dtype=bool)
    rows_ok[~same] = False
    inv = r["inv"].reshape(-1, k)
    tok_ok = rows_ok[inv].all(axis=1)
    _assert_close(out_gpu[tok_ok], r["out"][tok_ok], f"{what}: output of unaffected tokens")
    assert rel_out < LAYER_REL, f"{what}: layer output {rel_out:.3e}"


@pytest.mark.parametrize("tile_m", [128, 256, 1])
def test_nvfp4_grouped_fc1_swiglu_and_fc2(tile_m):
    shape = synth.scaled(synth.MOE_30B, T=300, H=512, I=256, E=6, k=4)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, pad=_pad(tile_m))
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    amax = torch.full((cap,), 7.0, dtype=torch.float32, device="cuda")    # gather zeroes it
    aq, as_, ats = ops.moe_gather_nvfp4(qx, sx, tsx, H, perm, seg, E, k, cap, amax_zero=amax)
    q1, s1, t1 = ops.nvfp4_quantize_weight([w1[:, :I].contiguous(), w1[:, I:].contiguous()])
    q2, s2, t2 = ops.nvfp4_quantize_weight([w2])
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         aq, q1.view(E * 2 * I, H // 2), as_, H // 16, s1, H // 16, d,
                         b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=t1, row_prob=rp,
                         out2=d, amax=amax, tile_m=tile_m)
    qd, sd, tsd = ops.nvfp4_quantize_per_token(d, amax_in=amax, m_valid=seg[E:])
    y = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                         qd, q2.view(E * H, I // 2), sd, I // 16, s2, I // 16, y,
                         b_rows_per_expert=H, alpha_a=tsd, alpha_b=t2, tile_m=tile_m)
    out = ops.moe_combine(y, inv, shape.T, k)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), E, pad=_pad(tile_m))
    R = int(r["seg"][-1])
    amax_ref = np.max(np.abs(np_bf16(d)[:R]), axis=1)
    assert np.array_equal(amax.cpu().numpy()[:R], amax_ref), "amax(D) equals the row max of D"
    _chained_compare(np_bf16(d), np_bf16(y), np_bf16(out), r, k, "NVFP4 layer")


@pytest.mark.parametrize("tile_m", [128, 256, 1])
def test_nvfp4_fc1_swiglu_extreme_gates(tile_m):
    """The SwiGLU epilogue where e^-g overflows or underflows fp32 and where
    g is tiny or exactly zero: tokens scaled by 1e-30, 1e-3, 1, 1e3 and 1e5
    (gate values from about 1e-35 to 2e5 in magnitude) and all-zero tokens.
    D stays finite, amax(D) is the row max of D, and D meets the oracle's
    fp64 SwiGLU within one bf16 step per element (or the row's floor).  Where
    g < -87.3 the helper's reciprocal of 1 + e^-g (above 2^126) flushes to
    zero, so D there is a zero, while the exact value is a tiny nonzero
    number (below 2^-119 |u| p); those elements are checked to be zero and
    are left out of the count of differing elements."""
    shape = synth.scaled(synth.MOE_30B, T=300, H=512, I=256, E=6, k=4)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, seed=3,
                                                                         pad=_pad(tile_m))
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    f = torch.tensor([1e-30, 1e-3, 1.0, 1e3, 1e5, 0.0], dtype=torch.float32)
    scale = f[torch.arange(shape.T) % f.numel()].cuda()[:, None]
    x = (x.float() * scale).to(torch.bfloat16).contiguous()
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    amax = torch.full((cap,), 7.0, dtype=torch.float32, device="cuda")
    aq, as_, ats = ops.moe_gather_nvfp4(qx, sx, tsx, H, perm, seg, E, k, cap, amax_zero=amax)
    q1, s1, t1 = ops.nvfp4_quantize_weight([w1[:, :I].contiguous(), w1[:, I:].contiguous()])
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         aq, q1.view(E * 2 * I, H // 2), as_, H // 16, s1, H // 16, d,
                         b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=t1, row_prob=rp,
                         out2=d, amax=amax, tile_m=tile_m)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), E, pad=_pad(tile_m))
    R = int(r["seg"][-1])
    g = r["acc1"][:R, :I]
    real = np.asarray(r["perm"])[:R] >= 0
    assert (np.abs(g[real]) > 88).any() and (np.abs(g[real][g[real] != 0]) < 1e-20).any(), \
        "the inputs reach both ends of the exponential's range"
    dk = np_bf16(d)[:R]
    assert np.all(np.isfinite(dk)), "D finite"
    assert np.array_equal(amax.cpu().numpy()[:R], np.max(np.abs(dk), axis=1)), "amax(D)"
    ref = r["d"]
    ulp = np.abs(ref) * 2.0 ** -7
    # rows of one token share a scale; the floor is relative to that row's largest value
    floor = 1e-4 * np.max(np.abs(ref), axis=1, keepdims=True)
    assert np.all(np.abs(dk - ref) <= np.maximum(ulp, floor)), "D beyond one bf16 step"
    flushed = g < -88.0
    assert np.all(dk[flushed & real[:, None]] == 0), "D is zero where the reciprocal flushes"
    assert np.all(np.abs(ref[flushed]) <= 2.0 ** -100 * np.abs(g[flushed]) *
                  np.abs(r["acc1"][:R, I:][flushed]) + 0.0), "the exact value there is tiny"
    ordinary = (np.abs(g) <= 87.0) & real[:, None]
    diff = (dk != ref)[ordinary]
    print(f"PARITY-STATS extreme gates tile_m {tile_m}: D elements differing {diff.mean():.3e} "
          f"of {diff.size} with |g| <= 87; {int(flushed.sum())} with g < -88 flushed to zero")
    assert diff.mean() < D_ELEM_DIFF, f"{diff.mean():.2e} of D elements differ"


def _fc1_by_flat_row(shape, tile_m):
    """FC1 (NVFP4, SwiGLU x prob epilogue) with the given GEMM kernel; D and
    amax(D) returned in routed-row order (token-major, slot-minor), which does
    not depend on the segment padding the kernel needs."""
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, pad=_pad(tile_m))
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    amax = torch.empty(cap, dtype=torch.float32, device="cuda")
    aq, as_, ats = ops.moe_gather_nvfp4(qx, sx, tsx, H, perm, seg, E, k, cap, amax_zero=amax)
    q1, s1, t1 = ops.nvfp4_quantize_weight([w1.contiguous()])
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         aq, q1.view(E * 2 * I, H // 2), as_, H // 16, s1, H // 16, d,
                         b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=t1, row_prob=rp,
                         out2=d, amax=amax, tile_m=tile_m)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    idx = inv.long()
    return d[idx].contiguous().view(torch.int16).cpu().numpy(), amax[idx].cpu().numpy()


@pytest.mark.parametrize("shape", [
    synth.scaled(synth.MOE_30B, T=300, H=512, I=256, E=6, k=4),
    synth.scaled(synth.MOE_30B, T=2048, E=32),
    synth.scaled(synth.MOE_671B, T=1024, E=16),
], ids=["small", "30b_H2048_I768", "671b_H7168_I2048"])
def test_nvfp4_fc1_identical_across_kernels(shape):
    """The one-CTA (128-row tiles), CTA-pair (256-row tiles) and small-M
    kernels give byte-identical D and amax(D) for every routed row: one
    activation definition in every epilogue, so which kernel runs (a choice
    made from the batch size) never changes the FP4 re-quantisation."""
    ref_d, ref_a = _fc1_by_flat_row(shape, 128)
    for tile_m in (256, 1):
        d, a = _fc1_by_flat_row(shape, tile_m)
        bad = np.flatnonzero((d != ref_d).any(axis=1))
        assert bad.size == 0, (f"tile_m {tile_m}: {bad.size} of {d.shape[0]} D rows differ from "
                               f"the one-CTA kernel's (first routed row {bad[0]})")
        assert np.array_equal(a.view(np.uint32), ref_a.view(np.uint32)), f"tile_m {tile_m}: amax"


@pytest.mark.parametrize("epi", ["bf16", "f32"])
def test_small_m_row_map_leaves_padding_rows(epi):
    """With the segment build's row map, the small-M kernel writes exactly
    the routed rows: they are byte-identical to the same GEMM without the
    map, and every padding row (row map < 0) keeps the sentinel the output
    buffer held.  Few tokens over many experts, so most rows are padding."""
    shape = synth.scaled(synth.MOE_30B, T=48, H=512, I=256, E=24, k=4)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, seed=5, pad=128)
    E, H, I = shape.E, shape.H, shape.I
    dsrc = synth.normal_bf16(5, 78, (cap, I), "cuda", std=0.05)
    qd, sd, tsd = ops.nvfp4_quantize_per_token(dsrc)
    q2, s2, t2 = ops.nvfp4_quantize_weight([w2])
    dt = torch.bfloat16 if epi == "bf16" else torch.float32
    code = L.EPI_BF16 if epi == "bf16" else L.EPI_F32
    outs = []
    for row_perm in (None, perm):
        y = torch.full((cap, H), -7.0, dtype=dt, device="cuda")
        ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, code, E, cap, H, I, seg,
                             qd, q2.view(E * H, I // 2), sd, I // 16, s2, I // 16, y,
                             b_rows_per_expert=H, alpha_a=tsd, alpha_b=t2,
                             tile_m=L.TILE_SMALL_M, row_perm=row_perm)
        outs.append(y)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    R = int(seg[-1].item())
    real = torch.zeros(cap, dtype=torch.bool, device="cuda")
    real[:R] = perm[:R] >= 0
    pad = ~real
    pad[R:] = False
    assert int(pad.sum()) > R // 2, "the case should be mostly padding"
    assert torch.equal(outs[1][real], outs[0][real]), "routed rows"
    assert bool((outs[1][pad] == -7.0).all()), "padding rows written"
    assert not bool((outs[0][pad] == -7.0).all()), "without the map every row is written"


@pytest.mark.parametrize("tile_m", [128, 256, 1])
def test_nvfp4_fc2_on_identical_operands(tile_m):
    """FC2 alone: the same seeded bf16 D quantised by both sides (byte-exact),
    then the grouped GEMM against the fp64 GEMM: strict tolerance."""
    shape = synth.scaled(synth.MOE_30B, T=400, H=768, I=512, E=5, k=3)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, seed=2, pad=_pad(tile_m))
    E, H, I = shape.E, shape.H, shape.I
    dsrc = synth.normal_bf16(2, 77, (cap, I), "cuda", std=0.05, outlier_p=1e-3, outlier_mul=20.0)
    qd, sd, tsd = ops.nvfp4_quantize_per_token(dsrc)
    q2, s2, t2 = ops.nvfp4_quantize_weight([w2])
    y = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                         qd, q2.view(E * H, I // 2), sd, I // 16, s2, I // 16, y,
                         b_rows_per_expert=H, alpha_a=tsd, alpha_b=t2, tile_m=tile_m)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    segn = seg.cpu().numpy()
    R = int(segn[-1])
    dn = np_bf16(dsrc)[:R]
    rq, rs, rts = Q.nvfp4_quantize_per_token(dn)
    a = Q.nvfp4_dequantize(rq, rs, rts)
    w2q = Q.nvfp4_quantize_joint([np_bf16(w2)], E)
    b = MO.dequant_weights_nvfp4(w2q)
    ref = F.bf16_round(MO.grouped_gemm(a, b, segn))
    _assert_close(np_bf16(y)[:R], ref, "NVFP4 FC2 (identical operands)")


@pytest.mark.parametrize("tile_m", [128, 256, 1])
def test_nvfp4_layer_api(tile_m):
    """The public layer API (NVFP4MoE) on a reduced 30B-A3B-shaped layer."""
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    shape = synth.scaled(synth.MOE_30B, T=512, H=1024, I=256, E=16)
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    layer = NVFP4MoE(shape.T, shape.H, shape.I, shape.E, shape.k, tile_m=tile_m)
    w = NVFP4Weights.quantize(w1, w2)
    out = layer.forward(x, ids.cuda(), prob.cuda(), w).clone()
    out2 = layer.forward(x, ids.cuda(), prob.cuda(), w)
    torch.cuda.synchronize()
    assert torch.equal(out, out2), "deterministic"
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), shape.E, pad=_pad(tile_m))
    _chained_compare(np_bf16(layer.d), np_bf16(layer.y), np_bf16(out), r, shape.k, "NVFP4MoE")


def test_nvfp4_layer_chunked_output():
    """forward(out_chunks=n, on_chunk=...) combines the output in n token
    ranges that tile [0, T) in order, each announced right after its launch,
    and gives the same bytes as one combine (T = 509 does not divide)."""
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    shape = synth.scaled(synth.MOE_30B, T=509, H=1024, I=256, E=16)
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    layer = NVFP4MoE(shape.T, shape.H, shape.I, shape.E, shape.k)
    w = NVFP4Weights.quantize(w1, w2)
    ref = layer.forward(x, ids.cuda(), prob.cuda(), w).clone()
    ranges = []
    out = torch.full_like(ref, float("nan"))
    layer.forward(x, ids.cuda(), prob.cuda(), w, out=out, out_chunks=5,
                  on_chunk=lambda j, t0, t1: ranges.append((j, t0, t1)))
    torch.cuda.synchronize()
    assert [r[0] for r in ranges] == list(range(5))
    assert ranges[0][1] == 0 and ranges[-1][2] == shape.T
    assert all(ranges[i][2] == ranges[i + 1][1] for i in range(4))
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("tile_m", [128, 256])
def test_mxfp8_grouped_fprop_dgrad_wgrad(tile_m):
    shape = synth.scaled(synth.MOE_30B_BWD, T=256, H=256, I=256, E=4, k=2)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, pad=tile_m)
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    xp = ops.moe_gather_bf16(x, perm, seg, E, k, cap)
    mx = ops.mxfp8_quantize(xp, m_valid=seg[E:])
    # fprop: Y = X_perm . W_e^T with W [E*256, H] (row-wise copies)
    w = synth.normal_bf16(9, 99, (E * 256, H), "cuda", std=0.02)
    wq = ops.mxfp8_quantize(w)
    y = torch.empty(cap, 256, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, 256, H, seg,
                         mx["row_q"], wq["row_q"], mx["row_s"], H // 32, wq["row_s"], H // 32,
                         y, b_rows_per_expert=256, tile_m=tile_m)
    # dgrad: dX = G . W_e with the column-wise copy of W ([H, E*256], stored transposed)
    gy = synth.normal_bf16(9, 98, (cap, 256), "cuda", std=1e-3)
    gq = ops.mxfp8_quantize(gy, colwise=False)
    dx = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, H, 256, seg,
                         gq["row_q"], wq["col_q"], gq["row_s"], 256 // 32, wq["col_s"],
                         (E * 256) // 32, dx, b_rows_per_expert=0, b_k_per_expert=256,
                         tile_m=tile_m)
    # wgrad: dW_e = gy_e^T . X_e over each expert's rows (column-wise copies)
    gc = ops.mxfp8_quantize(gy, rowwise=False, m_valid=seg[E:])
    dw = torch.empty(E, 256, H, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_K, L.EPI_F32, E, 256, H, 0, seg,
                         gc["col_q"], mx["col_q"], gc["col_s"], cap // 32, mx["col_s"],
                         cap // 32, dw, tile_m=tile_m)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    segn = seg.cpu().numpy()
    R = int(segn[-1])
    xpn = np_bf16(xp)[:R]
    wn = np_bf16(w).reshape(E, 256, H)
    gyn = np_bf16(gy)[:R]
    # fprop reference
    a = MO.mx_rows(xpn)
    b = np.stack([MO.mx_rows(wn[e]) for e in range(E)])
    _assert_close(np_bf16(y)[:R], F.bf16_round(MO.grouped_gemm(a, b, segn)), "MXFP8 fprop")
    # dgrad reference: B_e = column-wise copy of W_e ([H, 256] after transpose)
    wc = MO.mx_cols_t(np_bf16(w))                                   # [H, E*256]
    bd = np.stack([wc[:, e * 256:(e + 1) * 256] for e in range(E)])
    _assert_close(np_bf16(dx)[:R], F.bf16_round(MO.grouped_gemm(MO.mx_rows(gyn), bd, segn)),
                  "MXFP8 dgrad")
    ref_dw = MO.grouped_wgrad(MO.mx_cols_t(gyn), MO.mx_cols_t(xpn), segn)
    _assert_close(dw.cpu().numpy(), ref_dw, "MXFP8 wgrad")


@pytest.mark.parametrize("empty", [False, True])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_mxfp8_layer_fwd_bwd_api(tile_m, empty):
    """The MXFP8 layer (forward and backward) through MXFP8MoE against the
    oracle.  FC1's outputs (C = gate|up, D) come from identical operands and
    meet the GEMM tolerance; later stages consume re-quantised tensors, so a
    one-step bf16 difference upstream can move an E4M3 code: their bound is
    the same GEMM tolerance (measured errors are near 1e-5).  With ``empty``
    experts 0, 3 and 7 receive no rows: their weight gradients are zero."""
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    shape = synth.scaled(synth.MOE_30B_BWD, T=384, H=512, I=256, E=8, k=4)
    if empty:
        ids5, prob = synth.routing(synth.scaled(shape, E=5))
        ids = torch.tensor([1, 2, 4, 5, 6], dtype=torch.int32)[ids5.long()]
    else:
        ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    layer = MXFP8MoE(shape.T, shape.H, shape.I, shape.E, shape.k, tile_m=tile_m)
    layer.quantize_weights(w1, w2)
    out = layer.forward(x, ids.cuda(), prob.cuda())
    dx, dw1, dw2 = layer.backward(dy)
    torch.cuda.synchronize()
    from microscaled_precision_moe_gb300 import ops
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.mxfp8_moe_fwd_bwd(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), np_bf16(dy), shape.E, pad=tile_m)
    R = int(r["seg"][-1])
    if empty:
        segh = r["seg"]
        assert segh[1] == segh[0] and segh[4] == segh[3] and segh[8] == segh[7]
        assert not dw1[[0, 3, 7]].any() and not dw2[[0, 3, 7]].any()
    _assert_close(np_bf16(layer.c1)[:R], r["c1"], "MXFP8 FC1 C")
    _assert_close(np_bf16(layer.d)[:R], r["d"], "MXFP8 FC1 D")
    report = {}
    for name, got, ref in [("out", np_bf16(out), r["out"]), ("dh", np_bf16(layer.dh)[:R], r["dh"]),
                           ("dx", np_bf16(dx), r["dx"]), ("dw1", dw1.cpu().numpy(), r["dw1"]),
                           ("dw2", dw2.cpu().numpy(), r["dw2"])]:
        ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, REL, ELEM)
        report[name] = (rf, mx / max(bound / ELEM, 1e-30))
        assert ok, f"MXFP8 {name}: rel_frob={rf:.3e} max_err/max={mx / (bound / ELEM):.3e}"
    print("MXFP8 chained errors (rel_frob, max_err/max):", report)


def test_mxfp8_dswiglu_identical_across_kernels():
    """The SwiGLU backward fused into the FC2 dgrad gives the same dH bits on
    the one-CTA kernel (128-row segments) and on the CTA-pair kernel
    (256-row segments, two columns per packed f32x2 operation): the row-wise
    operands of each routed row are the same in both layouts, so every routed
    row's dgrad accumulator and epilogue inputs are too."""
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    shape = synth.scaled(synth.MOE_30B_BWD, T=384, H=512, I=768, E=8, k=4)
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    got = {}
    for tm in (128, 256):
        layer = MXFP8MoE(shape.T, shape.H, shape.I, shape.E, shape.k, tile_m=tm)
        layer.quantize_weights(w1, w2)
        layer.forward(x, ids.cuda(), prob.cuda())
        layer.backward(dy)
        torch.cuda.synchronize()
        inv = layer.seg[2].long()
        got[tm] = (layer.c1[inv].cpu(), layer.dh[inv].cpu())
    assert torch.equal(got[128][0], got[256][0]), "C = gate|up differs between kernels"
    same = (got[128][1] == got[256][1]).all(dim=1)
    assert bool(same.all()), f"dH differs on {int((~same).sum())} of {same.numel()} routed rows"


def test_mxfp8_fprop_small_m():
    """MXFP8 fprop (bf16 and fp32 out) and the SwiGLU epilogue on the small-M
    kernel: few rows per expert (decode-sized segments)."""
    shape = synth.scaled(synth.MOE_30B_BWD, T=40, H=512, I=256, E=8, k=2)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape, pad=128)
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    xp = ops.moe_gather_bf16(x, perm, seg, E, k, cap)
    mx = ops.mxfp8_quantize(xp, colwise=False, m_valid=seg[E:])
    w = synth.normal_bf16(9, 97, (E * 2 * I, H), "cuda", std=0.02)
    wq = ops.mxfp8_quantize(w, colwise=False)
    segn = seg.cpu().numpy()
    R = int(segn[-1])
    a = MO.mx_rows(np_bf16(xp)[:R])
    b = np.stack([MO.mx_rows(np_bf16(w).reshape(E, 2 * I, H)[e]) for e in range(E)])
    ref = MO.grouped_gemm(a, b, segn)
    for epi, dt in [(L.EPI_BF16, torch.bfloat16), (L.EPI_F32, torch.float32)]:
        y = torch.empty(cap, 2 * I, dtype=dt, device="cuda")
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, epi, E, cap, 2 * I, H, seg,
                             mx["row_q"], wq["row_q"], mx["row_s"], H // 32, wq["row_s"], H // 32,
                             y, b_rows_per_expert=2 * I, tile_m=1)
        torch.cuda.synchronize()
        assert ops.get_device_status() == 0
        got = np_bf16(y)[:R] if dt == torch.bfloat16 else y[:R].cpu().numpy()
        _assert_close(got, F.bf16_round(ref) if dt == torch.bfloat16 else ref,
                      f"MXFP8 small-M fprop ({epi})")
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(cap, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         mx["row_q"], wq["row_q"], mx["row_s"], H // 32, wq["row_s"], H // 32,
                         d, b_rows_per_expert=2 * I, row_prob=rp, out2=d, amax=amax, tile_m=1)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        dref = MO.fc1_epilogue(ref, rp.cpu().numpy()[:R], I)
    _assert_close(np_bf16(d)[:R], dref, "MXFP8 small-M SwiGLU")
    assert np.array_equal(amax.cpu().numpy()[:R], np.max(np.abs(np_bf16(d)[:R]), axis=1))


@pytest.mark.parametrize("tile_m", [256, 1])
def test_nvfp4_grouped_with_empty_experts(tile_m):
    """Experts 0, 3 and 7 of 8 receive no rows (empty segments at the start,
    in the middle and at the end): the kernels' walk over the segment
    offsets skips them and the layer still matches the oracle."""
    base = synth.scaled(synth.MOE_30B, T=260, H=512, I=256, E=5, k=3)
    ids5, prob = synth.routing(base, 3)
    remap = torch.tensor([1, 2, 4, 5, 6], dtype=torch.int32)
    ids = remap[ids5.long()]
    E = 8
    shape = synth.scaled(synth.MOE_30B, T=260, H=512, I=256, E=E, k=3)
    ops, L = _ops(), _L()
    H, I, k = shape.H, shape.I, shape.k
    x = synth.moe_activations(shape, 3, device="cuda")
    w1, w2 = synth.moe_weights(shape, 3, device="cuda")
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=_pad(tile_m))
    segh = seg.cpu().numpy()
    assert segh[1] == segh[0] and segh[4] == segh[3] and segh[8] == segh[7]
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    amax = torch.full((cap,), 7.0, dtype=torch.float32, device="cuda")
    aq, as_, ats = ops.moe_gather_nvfp4(qx, sx, tsx, H, perm, seg, E, k, cap, amax_zero=amax)
    q1, s1, t1 = ops.nvfp4_quantize_weight([w1.contiguous()])
    q2, s2, t2 = ops.nvfp4_quantize_weight([w2])
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         aq, q1.view(E * 2 * I, H // 2), as_, H // 16, s1, H // 16, d,
                         b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=t1, row_prob=rp,
                         out2=d, amax=amax, tile_m=tile_m)
    qd, sd, tsd = ops.nvfp4_quantize_per_token(d, amax_in=amax, m_valid=seg[E:])
    y = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                         qd, q2.view(E * H, I // 2), sd, I // 16, s2, I // 16, y,
                         b_rows_per_expert=H, alpha_a=tsd, alpha_b=t2, tile_m=tile_m)
    out = ops.moe_combine(y, inv, shape.T, k)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), E, pad=_pad(tile_m))
    assert np.array_equal(r["seg"], segh)
    _chained_compare(np_bf16(d), np_bf16(y), np_bf16(out), r, k, "NVFP4 layer, empty experts")
