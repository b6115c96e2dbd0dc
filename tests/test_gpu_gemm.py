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


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _ops():
    from microscaled_precision_moe_gb300 import ops
    return ops


def _L():
    from microscaled_precision_moe_gb300 import _lib
    return _lib


def _assert_close(got, ref, what):
    ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, REL, ELEM)
    assert ok, f"{what}: rel_frob={rf:.3e} max_err={mx:.3e} bound={bound:.3e}"


def test_nvfp4_single_expert_gate_up():
    """128 x 2048 activations (0.1% x50 outliers) against jointly quantised
    768 x 2048 gate and up weights -> 128 x 1536 fp32."""
    ops, L = _ops(), _L()
    x, wg, wu = synth.single_expert_inputs(device="cuda")
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    qw, sw, tsw = ops.nvfp4_quantize_weight([wg[None].contiguous(), wu[None].contiguous()])
    out = torch.empty(128, 1536, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_F32, 1, 128, 1536, 2048, None,
                         qx, qw[0], sx, 128, sw, 128, out, alpha_a=tsx, alpha_b=tsw)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    ref = MO.nvfp4_gemm_single(np_bf16(x), np_bf16(wg), np_bf16(wu))["c"]
    _assert_close(out.cpu().numpy(), ref.astype(np.float32), "single-expert NVFP4")


def _grouped_nvfp4_setup(shape, seed=0):
    ops = _ops()
    ids, prob = synth.routing(shape, seed)
    x = synth.moe_activations(shape, seed, device="cuda")
    w1, w2 = synth.moe_weights(shape, seed, device="cuda")
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), shape.E)
    return ids, prob, x, w1, w2, seg, perm, inv, rp, cap


def test_nvfp4_grouped_fc1_swiglu_and_fc2():
    shape = synth.scaled(synth.MOE_30B, T=300, H=512, I=256, E=6, k=4)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape)
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    qx, sx, tsx = ops.nvfp4_quantize_per_token(x)
    aq, as_, ats = ops.moe_gather_nvfp4(qx, sx, tsx, H, perm, seg, E, k, cap)
    q1, s1, t1 = ops.nvfp4_quantize_weight([w1[:, :I].contiguous(), w1[:, I:].contiguous()])
    q2, s2, t2 = ops.nvfp4_quantize_weight([w2])
    d = torch.empty(cap, I, dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(cap, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_SWIGLU, E, cap, 2 * I, H, seg,
                         aq, q1.view(E * 2 * I, H // 2), as_, H // 16, s1, H // 16, d,
                         b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=t1, row_prob=rp,
                         out2=d, amax=amax)
    qd, sd, tsd = ops.nvfp4_quantize_per_token(d, amax_in=amax, m_valid=seg[E:])
    y = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                         qd, q2.view(E * H, I // 2), sd, I // 16, s2, I // 16, y,
                         b_rows_per_expert=H, alpha_a=tsd, alpha_b=t2)
    out = ops.moe_combine(y, inv, shape.T, k)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                 np_bf16(w2), E)
    R = int(r["seg"][-1])
    _assert_close(np_bf16(d)[:R], r["d"], "FC1 SwiGLU D")
    amax_ref = np.max(np.abs(np_bf16(d)[:R]), axis=1)
    assert np.array_equal(amax.cpu().numpy()[:R], amax_ref), "amax(D) equals the row max of D"
    _assert_close(np_bf16(y)[:R], r["y"], "FC2 Y_perm")
    _assert_close(np_bf16(out), r["out"], "layer output")


def test_mxfp8_grouped_fprop_dgrad_wgrad():
    shape = synth.scaled(synth.MOE_30B_BWD, T=256, H=256, I=256, E=4, k=2)
    ops, L = _ops(), _L()
    ids, prob, x, w1, w2, seg, perm, inv, rp, cap = _grouped_nvfp4_setup(shape)
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    xp = ops.moe_gather_bf16(x, perm, seg, E, k, cap)
    mx = ops.mxfp8_quantize(xp, m_valid=seg[E:])
    # fprop: Y = X_perm . W_e^T with W [E*256, H] (row-wise copies)
    w = synth.normal_bf16(9, 99, (E * 256, H), "cuda", std=0.02)
    wq = ops.mxfp8_quantize(w)
    y = torch.empty(cap, 256, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, 256, H, seg,
                         mx["row_q"], wq["row_q"], mx["row_s"], H // 32, wq["row_s"], H // 32,
                         y, b_rows_per_expert=256)
    # dgrad: dX = G . W_e with the column-wise copy of W ([H, E*256], stored transposed)
    gy = synth.normal_bf16(9, 98, (cap, 256), "cuda", std=1e-3)
    gq = ops.mxfp8_quantize(gy, colwise=False)
    dx = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, H, 256, seg,
                         gq["row_q"], wq["col_q"], gq["row_s"], 256 // 32, wq["col_s"],
                         (E * 256) // 32, dx, b_rows_per_expert=0, b_k_per_expert=256)
    # wgrad: dW_e = gy_e^T . X_e over each expert's rows (column-wise copies)
    gc = ops.mxfp8_quantize(gy, rowwise=False, m_valid=seg[E:])
    dw = torch.empty(E, 256, H, dtype=torch.float32, device="cuda")
    ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_K, L.EPI_F32, E, 256, H, 0, seg,
                         gc["col_q"], mx["col_q"], gc["col_s"], cap // 32, mx["col_s"],
                         cap // 32, dw)
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
