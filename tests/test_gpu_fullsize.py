"""Parity at the full workload sizes, in the launch configuration bench.py times
(CTA-pair GEMMs, 256-row segments).

The layers run whole on the GPU; the oracle recomputes sampled outputs one
expert at a time (it needs only the weights of the experts it checks):

* per-token codes / scales / token scales of sampled rows: byte-exact;
* segment offsets, permutation, inverse permutation: bit-exact (whole);
* FC1 output D on every routed row of the checked experts: GEMM tolerance;
* FC2 output Y on those rows whose D is bit-identical to the oracle's (so the
  re-quantised operands are identical): GEMM tolerance; other rows within
  the NVFP4 re-quantisation noise;
* combine: the output equals, bit for bit, the oracle's combine of the
  kernel's own Y rows (fetched a chunk of tokens at a time, so it holds at
  any size);
* MXFP8 forward and backward: X and dY quantised into the checked experts'
  rows (row-wise and column-wise codes, column scales): byte-exact; C, D, Y,
  dH rows and the full dW1 / dW2 of the checked experts: GEMM tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q
from oracle import moe as MO
from oracle import metrics as Mx
from microscaled_precision_moe_gb300 import synth
from tests.gpu_util import need_gpu, np_bf16, u8, assert_bytes_equal, oracle_combine_check

pytestmark = pytest.mark.gpu

REL, ELEM = 1e-3, 1e-2
# chained NVFP4 bounds (see tests/test_gpu_gemm.py), per checked expert:
# fraction of D rows that differ from the oracle's and relative error of Y on
# those rows.  Measured on GB300 at these sizes: at most 3.8 % of the rows of
# the heaviest or middle expert differ (7.7 %, 4 of 52 rows, on the smallest
# decode batch) and their Y is within 1.4e-2.
D_ROW_DIFF = 0.15
REQUANT_REL = 0.05


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _close(got, ref, what, rel=REL, elem=ELEM):
    ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, rel, elem)
    assert ok, f"{what}: rel_frob={rf:.3e} max_err={mx:.3e} bound={bound:.3e}"


def _pick_experts(seg, n):
    """The heaviest, the lightest non-empty and a middle expert (n total)."""
    sizes = np.diff(seg)
    nz = np.flatnonzero(sizes > 0)
    order = nz[np.argsort(sizes[nz], kind="stable")]
    picks = [int(order[-1]), int(order[0])]
    mid = order[len(order) // 2:]
    for e in mid:
        if len(picks) >= n:
            break
        if int(e) not in picks:
            picks.append(int(e))
    return picks


def _nvfp4_expert_reference(xn_rows, w1e, w2e, prob, I):
    """Oracle NVFP4 path for the rows of one expert: per-token X quantisation,
    joint gate/up and W2 quantisation, fp64 FC1, SwiGLU x prob -> bf16 D, row
    amax, re-quantisation, fp64 FC2 -> bf16 Y.  Also returns the expert's
    quantised W1 and W2 (codes, block scales, outer scale)."""
    qx, sx, tsx = Q.nvfp4_quantize_per_token(xn_rows)
    a = Q.nvfp4_dequantize(qx, sx, tsx)
    w1q = Q.nvfp4_quantize_joint([w1e[None, :I], w1e[None, I:]], 1)
    w2q = Q.nvfp4_quantize_joint([w2e[None]], 1)
    b1 = MO.dequant_weights_nvfp4(w1q)[0]
    b2 = MO.dequant_weights_nvfp4(w2q)[0]
    with np.errstate(over="ignore"):
        d = MO.fc1_epilogue(a @ b1.T, prob, I)
    amax = np.max(np.abs(d), axis=1).astype(np.float32)
    qd, sd, tsd = Q.nvfp4_quantize_per_token(d, amax)
    y = F.bf16_round(Q.nvfp4_dequantize(qd, sd, tsd) @ b2.T)
    return d, y, w1q, w2q


def _check_expert_weights(W, e, w1q, w2q, what):
    """The library's joint weight quantisation of expert e, byte for byte:
    codes, the expert's tiled block scales (each expert's rows are tiled on
    their own) and its outer scale, for W1 (gate|up) and W2."""
    for name, (q, s, ts), (rq, rs, rts) in (("W1", (W.w1_q, W.w1_s, W.w1_ts), w1q),
                                           ("W2", (W.w2_q, W.w2_s, W.w2_ts), w2q)):
        rows, kh = q.shape[1], q.shape[2]
        nsb = Q.scale_bytes(rows, kh // 8)
        assert_bytes_equal(u8(q[e]), rq[0], f"{what}: {name} codes")
        got_s = Q.unswizzle_scales(u8(s[e * nsb:(e + 1) * nsb]), rows, kh // 8)
        assert_bytes_equal(got_s, rs[0], f"{what}: {name} block scales")
        assert_bytes_equal(ts[e:e + 1].cpu().numpy().view(np.uint32), rts.view(np.uint32),
                           f"{what}: {name} outer scale")


def _run_nvfp4_full(shape, n_experts, x_rows_checked, tile_m=256):
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    layer = NVFP4MoE(shape.T, shape.H, shape.I, shape.E, shape.k, tile_m=tile_m)
    out = layer.forward(x, ids.cuda(), prob.cuda(), W)
    torch.cuda.synchronize()
    from microscaled_precision_moe_gb300 import ops
    assert ops.get_device_status() == 0
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    # segments, whole
    seg_g, perm_g, inv_g, rp_g = [t.cpu().numpy() for t in layer.seg]
    seg, perm, inv, rp = MO.build_segments(ids.numpy(), prob.numpy(), E, layer.pad)
    assert_bytes_equal(seg_g, seg, "seg_offsets")
    R = int(seg[-1])
    assert_bytes_equal(perm_g[:R], perm, "perm")
    assert_bytes_equal(inv_g, inv, "inv_perm")
    # per-token quantisation of sampled tokens, read at each token's first
    # routed row (the quantiser writes straight into the routed rows)
    rows = np.random.default_rng(1).choice(T, x_rows_checked, replace=False)
    xr = np_bf16(x[torch.from_numpy(rows).cuda()])
    rq, rs, rts = Q.nvfp4_quantize_per_token(xr)
    qx, sx, tsx = layer.aq
    dst = inv_g[rows * k]
    cap = qx.shape[0]
    assert_bytes_equal(u8(qx)[dst], rq, "X codes (sampled tokens)")
    assert_bytes_equal(Q.unswizzle_scales(u8(sx), cap, H // 16)[dst], rs, "X scales (sampled tokens)")
    assert_bytes_equal(tsx.cpu().numpy()[dst].view(np.uint32), rts.view(np.uint32), "X token scales")
    # combine on the whole output: the oracle's combine of the kernel's own Y
    # rows, bit for bit
    oracle_combine_check(out, layer.y, inv_g, T, k, "combine")
    # FC1 / FC2 on every routed row of the checked experts
    d_g = layer.d
    y_gpu = layer.y
    for e in _pick_experts(seg, n_experts):
        r0, r1 = int(seg[e]), int(seg[e + 1])
        real = perm[r0:r1] >= 0
        rws = np.arange(r0, r1)[real]
        toks = perm[rws] // k
        xe = np_bf16(x[torch.from_numpy(toks).cuda()])
        w1e = np_bf16(w1[e])
        w2e = np_bf16(w2[e])
        d_ref, y_ref, w1q, w2q = _nvfp4_expert_reference(xe, w1e, w2e, rp[rws], I)
        _check_expert_weights(W, e, w1q, w2q, f"expert {e}")
        d_got = np_bf16(d_g[torch.from_numpy(rws).cuda()])
        y_got = np_bf16(y_gpu[torch.from_numpy(rws).cuda()])
        _close(d_got, d_ref, f"expert {e} ({len(rws)} rows): FC1 D")
        same = (d_got == d_ref).all(axis=1)
        rel = 0.0
        if (~same).any():
            rel = float(np.linalg.norm(y_got[~same] - y_ref[~same]) / np.linalg.norm(y_ref[~same]))
        print(f"PARITY-STATS {shape.name} expert {e} ({len(rws)} rows): D elements differing "
              f"{(d_got != d_ref).mean():.3e}, D rows differing {1.0 - same.mean():.4f}, "
              f"re-quantised rows rel {rel:.3e}")
        assert 1.0 - same.mean() < D_ROW_DIFF, f"expert {e}: {1.0 - same.mean():.3f} of D rows differ"
        _close(y_got[same], y_ref[same], f"expert {e}: FC2 Y on identical operands")
        assert rel < REQUANT_REL, f"expert {e}: re-quantised rows differ by {rel:.3e}"


def test_nvfp4_layer_30b_full_size():
    """16384 tokens, hidden 2048, 128 experts, intermediate 768, top-8."""
    _run_nvfp4_full(synth.MOE_30B, n_experts=4, x_rows_checked=512)


def test_nvfp4_layer_671b_full_size():
    """The headline workload: 32768 tokens, hidden 7168, 256 experts,
    intermediate 2048, top-8 with Zipf(1.1) expert load."""
    _run_nvfp4_full(synth.MOE_671B, n_experts=3, x_rows_checked=256)


@pytest.mark.parametrize("T", [64, 256])
def test_nvfp4_layer_671b_decode_small_m(T):
    """Decode-sized batches of the 671B-shaped layer (64 and 256 tokens over
    256 experts, Zipf load) on the small-M kernel, the bench's decode launch
    configuration: full hidden / intermediate sizes, sampled experts."""
    from microscaled_precision_moe_gb300 import _lib as L
    _run_nvfp4_full(synth.scaled(synth.MOE_671B, T=T), n_experts=3, x_rows_checked=min(T, 64),
                    tile_m=L.TILE_SMALL_M)


def test_mxfp8_layer_30b_fwd_bwd_full_size():
    """8192 tokens, hidden 2048, 128 experts, intermediate 768, top-8:
    forward and backward, checked on every row and the full weight gradients
    of three experts."""
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    shape = synth.MOE_30B_BWD
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    L = MXFP8MoE(T, H, I, E, k)
    L.quantize_weights(w1, w2)
    L.forward(x, ids.cuda(), prob.cuda())
    dx, dw1, dw2 = L.backward(dy)
    torch.cuda.synchronize()
    from microscaled_precision_moe_gb300 import ops
    assert ops.get_device_status() == 0
    seg, perm, inv, rp = MO.build_segments(ids.numpy(), prob.numpy(), E, L.tile_m)
    assert_bytes_equal(L.seg[0].cpu().numpy(), seg, "seg_offsets")
    for e in _pick_experts(seg, 3):
        r0, r1 = int(seg[e]), int(seg[e + 1])
        rws = np.arange(r0, r1)
        real = perm[r0:r1] >= 0
        toks = np.where(real, perm[r0:r1] // k, 0)
        # the expert's slice of the permuted operands (padding rows zero)
        xe = np_bf16(x[torch.from_numpy(toks).cuda()]) * real[:, None]
        dye = np_bf16(dy[torch.from_numpy(toks).cuda()]) * real[:, None]
        w1e, w2e = np_bf16(w1[e]), np_bf16(w2[e])
        p = rp[r0:r1]
        segl = np.array([0, r1 - r0])
        with np.errstate(over="ignore"):
            acc1 = MO.grouped_gemm(MO.mx_rows(xe), MO.mx_rows(w1e)[None], segl)
            c1 = F.bf16_round(acc1)
            d = MO.fc1_epilogue(acc1, p, I)
            y = F.bf16_round(MO.grouped_gemm(MO.mx_rows(d), MO.mx_rows(w2e)[None], segl))
            dd = MO.grouped_gemm(MO.mx_rows(dye), MO.mx_cols_t(w2e)[None], segl)
            dh = F.bf16_round(MO.swiglu_backward(dd, c1, p, I))
            dxp = F.bf16_round(MO.grouped_gemm(MO.mx_rows(dh), MO.mx_cols_t(w1e)[None], segl))
            dw2e = MO.grouped_wgrad(MO.mx_cols_t(dye), MO.mx_cols_t(d), segl)[0]
            dw1e = MO.grouped_wgrad(MO.mx_cols_t(dh), MO.mx_cols_t(xe), segl)[0]
        sel = torch.from_numpy(rws).cuda()
        # X and dY quantised from the token rows into this expert's rows
        # (segments start on 256-row boundaries: whole column blocks), bytes
        for q, v, what in ((L.xq, xe, "X"), (L.dyq, dye, "dY")):
            v = np.where(real[:, None], v, 0.0)        # padding rows +0, as gathered
            rq, rs = Q.mxfp8_quantize_rowwise(v)
            assert_bytes_equal(u8(q["row_q"][sel]), rq, f"expert {e}: {what} row codes")
            cq, cs = Q.mxfp8_quantize_colwise(v)
            assert_bytes_equal(u8(q["col_q"][:, r0:r1]), cq, f"expert {e}: {what} column codes")
            got_cs = Q.unswizzle_scales(u8(q["col_s"]), H, (L.cap + 31) // 32)
            assert_bytes_equal(got_cs[:, r0 // 32:r1 // 32], cs, f"expert {e}: {what} column scales")
        _close(np_bf16(L.c1[sel]), c1, f"expert {e}: C = gate|up")
        _close(np_bf16(L.d[sel]), d, f"expert {e}: D")
        _close(np_bf16(L.y[sel]), y, f"expert {e}: Y")
        _close(np_bf16(L.dh[sel]), dh, f"expert {e}: dH")
        _close(np_bf16(L.dxp[sel]), dxp, f"expert {e}: dX_perm")
        _close(dw1[e].cpu().numpy(), dw1e, f"expert {e}: dW1")
        _close(dw2[e].cpu().numpy(), dw2e, f"expert {e}: dW2")
    # dX: the oracle's combine of the kernel's own dX_perm rows, whole
    oracle_combine_check(dx, L.dxp, L.seg[2].cpu().numpy(), T, k, "dX combine")


def _nvfp4_bf16_bwd_expert_reference(xe, w1e, w2e, dye, p, I, mode):
    """Oracle for the rows of one expert (padding rows zero): the NVFP4
    forward (per-token X, joint gate/up W1, W2; C = gate|up in bf16; D; the
    re-quantised D) and the BF16 backward on the operands of ``mode``."""
    qx, sx, tsx = Q.nvfp4_quantize_per_token(xe)
    w1q = Q.nvfp4_quantize_joint([w1e[None, :I], w1e[None, I:]], 1)
    w2q = Q.nvfp4_quantize_joint([w2e[None]], 1)
    with np.errstate(over="ignore"):
        acc1 = Q.nvfp4_dequantize(qx, sx, tsx) @ MO.dequant_weights_nvfp4(w1q)[0].T
    c1 = F.bf16_round(acc1)
    d = MO.fc1_epilogue(acc1, p, I)
    qd, sd, tsd = Q.nvfp4_quantize_per_token(d, np.max(np.abs(d), axis=1).astype(np.float32))
    if mode == "high_precision":
        xo, b1, b2, do = xe.astype(np.float64), w1e.astype(np.float64), w2e.astype(np.float64), d
    else:
        xo = Q.nvfp4_dequantize_bf16(qx, sx, tsx)
        b1 = Q.nvfp4_dequantize_bf16(w1q[0][0], w1q[1][0], w1q[2][0])
        b2 = Q.nvfp4_dequantize_bf16(w2q[0][0], w2q[1][0], w2q[2][0])
        do = Q.nvfp4_dequantize_bf16(qd, sd, tsd)
    segl = np.array([0, xe.shape[0]])
    r = MO.bf16_backward(xo, b1[None], b2[None], do, c1, dye.astype(np.float64), segl, p, I)
    r.update(c1=c1, d=d, d_op=do)
    return r


def test_nvfp4_layer_30b_bf16_backward_full_size():
    """8192 tokens, hidden 2048, 128 experts, intermediate 768, top-8: the
    NVFP4 forward saving gate|up, then the BF16 backward in both operand
    modes (the bench launch configuration), checked on every row and the
    full weight gradients of three experts; dX by the combine property."""
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    from microscaled_precision_moe_gb300 import ops
    shape = synth.MOE_30B_BWD
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    L = NVFP4MoE(T, H, I, E, k)
    L.forward(x, ids.cuda(), prob.cuda(), W, save_for_backward=True)
    seg, perm, inv, rp = MO.build_segments(ids.numpy(), prob.numpy(), E, L.tile_m)
    picks = _pick_experts(seg, 3)
    for mode in NVFP4MoE.BACKWARD_MODES:
        L.prepare_backward_weights(mode, w1=w1, w2=w2, w=W)
        dx, dw1, dw2 = L.backward(dy, mode, x=x)
        torch.cuda.synchronize()
        assert ops.get_device_status() == 0
        for e in picks:
            r0, r1 = int(seg[e]), int(seg[e + 1])
            rws = np.arange(r0, r1)
            real = perm[r0:r1] >= 0
            toks = np.where(real, perm[r0:r1] // k, 0)
            sel = torch.from_numpy(toks).cuda()
            xe = np_bf16(x[sel]) * real[:, None]
            dye = np_bf16(dy[sel]) * real[:, None]
            ref = _nvfp4_bf16_bwd_expert_reference(xe, np_bf16(w1[e]), np_bf16(w2[e]), dye,
                                                   rp[r0:r1], I, mode)
            gsel = torch.from_numpy(rws).cuda()
            _close(np_bf16(L.c1[gsel]), ref["c1"], f"{mode} expert {e}: C")
            _close(np_bf16(L.dh[gsel]), ref["dh"], f"{mode} expert {e}: dH")
            _close(np_bf16(L.dxp[gsel]), ref["dxp"], f"{mode} expert {e}: dX_perm")
            _close(dw1[e].cpu().numpy(), ref["dw1"][0], f"{mode} expert {e}: dW1")
            d_same = (np_bf16(L.d[gsel]) == ref["d"]).all(axis=1)
            if mode == "high_precision" or d_same.all():
                _close(dw2[e].cpu().numpy(), ref["dw2"][0], f"{mode} expert {e}: dW2")
            else:
                # re-quantised D rows that differ carry another FP4 encoding:
                # the GEMM against its own operands, then the noise band
                dop = np_bf16(L.dop[gsel]).astype(np.float64)
                assert np.array_equal(dop[d_same], ref["d_op"][d_same])
                _close(dw2[e].cpu().numpy(), dye.astype(np.float64).T @ dop,
                       f"{mode} expert {e}: dW2 on the kernel's own D_hat")
                assert Mx.rel_l2(dw2[e].cpu().numpy(), ref["dw2"][0]) < 0.05
        oracle_combine_check(dx, L.dxp, L.seg[2].cpu().numpy(), T, k, f"{mode}: dX combine")
