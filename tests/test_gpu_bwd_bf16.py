"""GPU parity of the BF16 backward path: dequantisation to bf16 and the bf16
transpose (bit-exact against the oracle), the kind::f16 CTA-pair grouped GEMM
(GEMM tolerance against fp64), and the NVFP4 layer's high-precision and
dequantized backward end to end.

Source of the path: "Towards Blackwell-native 8-bit and 4-bit RL", section
"High-precision and dequantized backward"."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q
from oracle import moe as MO
from oracle import metrics as Mx
from microscaled_precision_moe_gb300 import synth
from tests.gpu_util import need_gpu, np_bf16, u8, assert_bytes_equal

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


def _bits(t):
    """bf16 tensor -> uint16 bit patterns (numpy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _close(got, ref, what):
    ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, REL, ELEM)
    assert ok, f"{what}: rel_frob={rf:.3e} max_err={mx:.3e} bound={bound:.3e}"


# ------------------------------------------------------------------ dequantisation

@pytest.mark.parametrize("rows_per_outer", [1, 7])
def test_nvfp4_dequantize_random_codes(rows_per_outer):
    """Random codes, random E4M3 scales and outer scales spread over the
    whole fp32 range (subnormal ones included, plus a value whose fp32
    product lands on a bf16 tie): every element rounded once, bit-exact."""
    ops = _ops()
    rng = np.random.default_rng(11 + rows_per_outer)
    M, K = 300, 256                                    # ragged against 128-row tiles
    q = rng.integers(0, 256, size=(M, K // 2)).astype(np.uint8)
    sb = rng.integers(0, 0x7F, size=(M, K // 16)).astype(np.uint8)
    n_outer = -(-M // rows_per_outer)
    ex = rng.integers(-140, 100, size=n_outer)
    outer = np.ldexp(1.0 + rng.random(n_outer), ex).astype(np.float32)
    outer[0] = np.float32(1.0 + 109227 * 2.0 ** -23)  # double-rounding trap
    outer[1 % n_outer] = np.float32(2.0 ** -149)
    if rows_per_outer == 1:
        q[0, 0], sb[0, 0] = 0x03, 0x38                  # 1.5 * 1 * trap
    sg_rows = np.repeat(outer, rows_per_outer)[:M]
    ref = F.f64_to_bf16_bits(Q.nvfp4_dequantize(q, sb, sg_rows))
    if rows_per_outer == 1:
        assert F.bf16_bits_to_f32(ref[:1, :1])[0, 0] == 1.5234375
    out = torch.full((M, K + 8), -7.0, dtype=torch.bfloat16, device="cuda")
    ops.nvfp4_dequantize(torch.from_numpy(q).cuda(), torch.from_numpy(Q.swizzle_scales(sb)).cuda(),
                         torch.from_numpy(outer).cuda(), rows_per_outer, K, out=out[:, :K])
    torch.cuda.synchronize()
    assert_bytes_equal(_bits(out[:, :K]), ref, "NVFP4 -> bf16")
    assert torch.all(out[:, K:] == -7.0)


def test_nvfp4_dequantize_of_quantised_activations():
    """The per-token quantiser's own output (zero, subnormal-amax and large
    rows included), dequantised, against the oracle's quantise-dequantise;
    rows past the device row count stay untouched."""
    ops = _ops()
    x = synth.mxfp8_quantizer_input(M=512, K=512, device="cuda")
    M, K = x.shape
    q, s, ts = ops.nvfp4_quantize_per_token(x)
    mv = torch.tensor([M - 37], dtype=torch.int32, device="cuda")
    out = torch.full((M, K), 3.0, dtype=torch.bfloat16, device="cuda")
    ops.nvfp4_dequantize(q, s, ts, 1, K, m_valid=mv, out=out)
    torch.cuda.synchronize()
    rq, rs, rts = Q.nvfp4_quantize_per_token(np_bf16(x))
    ref = F.f64_to_bf16_bits(Q.nvfp4_dequantize(rq, rs, rts))
    assert_bytes_equal(_bits(out)[:M - 37], ref[:M - 37], "dequantised activations")
    assert torch.all(out[M - 37:] == 3.0)


def test_nvfp4_dequantize_weights_per_expert_scale():
    """Jointly quantised expert weights: one outer scale per expert
    (rows_per_outer = rows of one expert)."""
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=64, H=256, I=128, E=3, k=2)
    w1, _ = synth.moe_weights(shape, device="cuda")
    E, I2, H = w1.shape
    q, s, ts = ops.nvfp4_quantize_weight([w1.contiguous()])
    out = ops.nvfp4_dequantize(q.view(E * I2, H // 2), s, ts, I2, H)
    torch.cuda.synchronize()
    rp, rs, rg = Q.nvfp4_quantize_joint([np_bf16(w1)], E)
    ref = np.concatenate([F.f64_to_bf16_bits(Q.nvfp4_dequantize(rp[e], rs[e], rg[e]))
                          for e in range(E)])
    assert_bytes_equal(_bits(out), ref, "dequantised weights")


def test_mxfp8_dequantize():
    """Row-wise MXFP8 codes of the quantiser workload (zero, +-448 and
    subnormal rows included) and random codes with scale bytes near 0."""
    ops = _ops()
    x = synth.mxfp8_quantizer_input(M=384, K=512, device="cuda")
    M, K = x.shape
    o = ops.mxfp8_quantize(x, colwise=False)
    out = ops.mxfp8_dequantize(o["row_q"], o["row_s"])
    torch.cuda.synchronize()
    c, sc = Q.mxfp8_quantize_rowwise(np_bf16(x))
    with np.errstate(over="ignore"):
        ref = F.f64_to_bf16_bits(Q.mxfp8_dequantize(c, sc))
    assert_bytes_equal(_bits(out), ref, "MXFP8 -> bf16")
    rng = np.random.default_rng(3)
    c = rng.integers(0, 256, size=(130, 96)).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x11
    sc = rng.integers(0, 12, size=(130, 3)).astype(np.uint8)
    sc[::3] = rng.integers(100, 255, size=(44, 3))
    out = ops.mxfp8_dequantize(torch.from_numpy(c).cuda(), torch.from_numpy(Q.swizzle_scales(sc)).cuda())
    torch.cuda.synchronize()
    with np.errstate(over="ignore"):
        ref = F.f64_to_bf16_bits(Q.mxfp8_dequantize(c, sc))
    assert_bytes_equal(_bits(out), ref, "MXFP8 extremes")


@pytest.mark.parametrize("R,C,ldi,valid", [(333, 200, 208, None), (64, 64, 64, 64),
                                           (1000, 72, 80, 777), (1, 8, 8, None)])
def test_transpose_bf16(R, C, ldi, valid):
    ops = _ops()
    base = synth.normal_bf16(5, 77, (R, ldi), device="cuda")
    x = base[:, :C]
    out = torch.full((C, R + 16), 9.0, dtype=torch.bfloat16, device="cuda")
    mv = None if valid is None else torch.tensor([valid], dtype=torch.int32, device="cuda")
    ops.transpose_bf16(x, m_valid=mv, out=out[:, :R])
    torch.cuda.synchronize()
    Rv = R if valid is None else valid
    ref = _bits(x).T
    assert_bytes_equal(_bits(out[:, :Rv]), ref[:, :Rv], "transpose")
    assert torch.all(out[:, Rv:] == 9.0)


# ------------------------------------------------------------------ BF16 grouped GEMM

def _segments(T, E, k, seed, skew=False):
    ops = _ops()
    shape = synth.scaled(synth.MOE_671B if skew else synth.MOE_30B, T=T, H=256, I=256, E=E, k=k)
    ids, prob = synth.routing(shape, seed)
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=256)
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), E, 256)
    return seg, rp, cap, rseg, rrp


def _bf16_rows(seed, tid, rows, cols, real_rows=None, std=1.0):
    t = synth.normal_bf16(seed, tid, (rows, cols), device="cuda", std=std)
    if real_rows is not None:
        t[real_rows:] = 0
    return t


@pytest.mark.parametrize("epi", ["bf16", "f32"])
def test_bf16_grouped_gemm_group_m(epi):
    """Expert segments of 256-row multiples; B addressed per expert by row
    offset (fprop layout) and by reduction offset (dgrad layout)."""
    ops, L = _ops(), _L()
    E, N, K = 5, 512, 384
    seg, rp, cap, rseg, _ = _segments(700, E, 3, 1)
    R = int(rseg[-1])
    a = _bf16_rows(1, 1, cap, K, R)
    b = _bf16_rows(1, 2, E * N, K, std=0.05)
    kind = L.KIND_BF16
    if epi == "bf16":
        out = torch.empty(cap, N, dtype=torch.bfloat16, device="cuda")
        ops.moe_grouped_gemm(kind, L.GROUP_M, L.EPI_BF16, E, cap, N, K, seg, a, b, None, 0, None, 0,
                             out, b_rows_per_expert=N, tile_m=256)
    else:
        out = torch.empty(cap, N, dtype=torch.float32, device="cuda")
        ops.moe_grouped_gemm(kind, L.GROUP_M, L.EPI_F32, E, cap, N, K, seg, a, b, None, 0, None, 0,
                             out, b_rows_per_expert=N, tile_m=256)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    an = np_bf16(a).astype(np.float64)
    bn = np_bf16(b).astype(np.float64).reshape(E, N, K)
    ref = MO.grouped_gemm(an[:R], bn, rseg)
    got = np_bf16(out[:R]) if epi == "bf16" else out[:R].cpu().numpy()
    _close(got, F.bf16_round(ref) if epi == "bf16" else ref, f"BF16 GROUP_M ({epi})")
    # the same GEMM with B given as a transposed copy [K, E*N]^T -> K-major
    # rows [N, E*K]: expert e's reduction columns start at e*K
    bt = torch.cat([b[e * N:(e + 1) * N] for e in range(E)], dim=1).contiguous()   # [N, E*K]
    out2 = torch.empty(cap, N, dtype=torch.bfloat16, device="cuda")
    ops.moe_grouped_gemm(kind, L.GROUP_M, L.EPI_BF16, E, cap, N, K, seg, a, bt, None, 0, None, 0,
                         out2, b_rows_per_expert=0, b_k_per_expert=K, tile_m=256)
    torch.cuda.synchronize()
    _close(np_bf16(out2[:R]), F.bf16_round(ref), "BF16 GROUP_M, reduction-offset B")
    # B stored MN-major: [E*K, N], expert e's reduction rows at e*K
    bmn = torch.cat([b[e * N:(e + 1) * N].t() for e in range(E)], dim=0).contiguous()
    out3 = torch.empty(cap, N, dtype=out.dtype, device="cuda")
    ops.moe_grouped_gemm(kind, L.GROUP_M, L.EPI_BF16 if epi == "bf16" else L.EPI_F32, E, cap, N, K,
                         seg, a, bmn, None, 0, None, 0, out3, b_rows_per_expert=0,
                         b_k_per_expert=K, tile_m=256, b_mn_major=True)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    got3 = np_bf16(out3[:R]) if epi == "bf16" else out3[:R].cpu().numpy()
    _close(got3, F.bf16_round(ref) if epi == "bf16" else ref, f"BF16 GROUP_M, MN-major B ({epi})")


@pytest.mark.parametrize("b_mn", [False, True])
def test_bf16_grouped_gemm_dswiglu(b_mn):
    """dH = SwiGLU backward of dD = dY W2 (W2 as a transposed copy, or read
    row-major as stored), with gate|up read from C."""
    ops, L = _ops(), _L()
    E, I, H = 4, 256, 512
    seg, rp, cap, rseg, rrp = _segments(500, E, 2, 2)
    R = int(rseg[-1])
    dy = _bf16_rows(2, 3, cap, H, R, std=1e-3)
    w2t = _bf16_rows(2, 4, I, E * H, std=0.05)           # [I, E*H]
    c1 = _bf16_rows(2, 5, cap, 2 * I, R)
    dh = torch.empty(cap, 2 * I, dtype=torch.bfloat16, device="cuda")
    bop = w2t.t().contiguous() if b_mn else w2t          # W2 as stored: [E*H, I]
    ops.moe_grouped_gemm(L.KIND_BF16, L.GROUP_M, L.EPI_DSWIGLU, E, cap, I, H, seg, dy, bop,
                         None, 0, None, 0, dh, b_rows_per_expert=0, b_k_per_expert=H,
                         row_prob=rp, aux=c1, tile_m=256, b_mn_major=b_mn)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    w2 = np_bf16(w2t).astype(np.float64).reshape(I, E, H).transpose(1, 0, 2)   # [E, I, H]
    dd = MO.grouped_gemm(np_bf16(dy).astype(np.float64)[:R], w2, rseg)
    ref = F.bf16_round(MO.swiglu_backward(dd, np_bf16(c1).astype(np.float64)[:R], rrp, I))
    _close(np_bf16(dh[:R]), ref, "BF16 dgrad + SwiGLU backward")


@pytest.mark.parametrize("mn", [False, True])
def test_bf16_grouped_gemm_group_k(mn):
    """Weight gradient: contraction over each expert's rows (an empty
    expert gives zeros), fp32 output per expert; operands as transposed
    copies, or read row-major as the layer holds them (MN-major)."""
    ops, L = _ops(), _L()
    E, Mo, N = 6, 512, 256
    shape = synth.scaled(synth.MOE_30B, T=400, H=256, I=256, E=E, k=2)
    ids, prob = synth.routing(shape, 4)
    ids = ids.clone()
    ids[ids == 2] = 3                                    # expert 2 gets no rows
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=256)
    rseg = MO.build_segments(ids.numpy(), prob.numpy(), E, 256)[0]
    assert rseg[3] == rseg[2]
    R = int(rseg[-1])
    at = _bf16_rows(4, 6, Mo, cap)
    bt = _bf16_rows(4, 7, N, cap)
    at[:, R:] = 0
    bt[:, R:] = 0
    out = torch.full((E, Mo, N), 5.0, dtype=torch.float32, device="cuda")
    aop, bop = (at.t().contiguous(), bt.t().contiguous()) if mn else (at, bt)
    ops.moe_grouped_gemm(L.KIND_BF16, L.GROUP_K, L.EPI_F32, E, Mo, N, 0, seg, aop, bop,
                         None, 0, None, 0, out, tile_m=256, a_mn_major=mn, b_mn_major=mn)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    ref = MO.grouped_wgrad(np_bf16(at).astype(np.float64), np_bf16(bt).astype(np.float64), rseg)
    got = out.cpu().numpy()
    assert np.all(got[2] == 0.0)
    _close(got, ref, "BF16 GROUP_K wgrad")


# ------------------------------------------------------------------ NVFP4 layer, BF16 backward

@pytest.mark.parametrize("mode", ["high_precision", "dequantized"])
def test_nvfp4_layer_bf16_backward(mode):
    """Forward (saving gate|up), then the BF16 backward in each operand mode,
    against the oracle's NVFP4 forward + BF16 backward.  Operands that come
    from the forward's re-quantised D are compared where the kernel's D
    equals the oracle's D bit for bit (the FP4 re-quantisation is
    discontinuous); everything else meets the GEMM tolerance whole."""
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=600, H=512, I=256, E=6, k=4)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    layer = NVFP4MoE(T, H, I, E, k)
    layer.forward(x, ids.cuda(), prob.cuda(), W, save_for_backward=True)
    layer.prepare_backward_weights(mode, w1=w1, w2=w2, w=W)
    dx, dw1, dw2 = layer.backward(dy, mode, x=x)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    xn, dyn = np_bf16(x).astype(np.float64), np_bf16(dy).astype(np.float64)
    w1n, w2n = np_bf16(w1).astype(np.float64), np_bf16(w2).astype(np.float64)
    with np.errstate(over="ignore"):
        fwd = MO.nvfp4_moe_forward(xn, ids.numpy(), prob.numpy(), w1n, w2n, E, pad=256)
        r = MO.nvfp4_moe_backward_bf16(fwd, xn, w1n, w2n, dyn, mode)
    R = int(fwd["seg"][-1])
    _close(np_bf16(layer.c1[:R]), r["c1"], "C = gate|up")
    d_same = (np_bf16(layer.d[:R]) == fwd["d"]).all(axis=1)
    assert d_same.mean() > 0.9
    if mode == "dequantized":
        assert_bytes_equal(_bits(layer.xp[:R]), F.f64_to_bf16_bits(r["xp"]), "X_hat (gathered)")
        dop = np_bf16(layer.dop[:R])
        assert np.array_equal(dop[d_same], r["d_op"][d_same]), "D_hat on identical D rows"
    else:
        assert_bytes_equal(_bits(layer.xp[:R]), F.f64_to_bf16_bits(r["xp"]), "X (gathered)")
    _close(np_bf16(layer.dh[:R]), r["dh"], f"{mode}: dH")
    _close(np_bf16(layer.dxp[:R]), r["dxp"], f"{mode}: dX_perm")
    _close(np_bf16(dx), r["dx"], f"{mode}: dX")
    _close(dw1.cpu().numpy(), r["dw1"], f"{mode}: dW1")
    if mode == "high_precision" or d_same.all():
        _close(dw2.cpu().numpy(), r["dw2"], f"{mode}: dW2")
    else:
        # dW2 contracts the re-quantised D_hat: rows whose D differs by a bf16
        # step carry another FP4 encoding.  The GEMM itself meets the
        # tolerance on the operands it was given (a property of the kernel's
        # own output, checked with plain numpy), and the result stays within
        # the re-quantisation noise of the oracle's.
        seg = fwd["seg"]
        dyp = np_bf16(layer.dyp[:R]).astype(np.float64)
        assert np.array_equal(dyp, r["dyp"])
        dop = np_bf16(layer.dop[:R]).astype(np.float64)
        own = np.stack([dyp[seg[e]:seg[e + 1]].T @ dop[seg[e]:seg[e + 1]] for e in range(E)])
        _close(dw2.cpu().numpy(), own, f"{mode}: dW2 on the kernel's own D_hat")
        rel = Mx.rel_l2(dw2.cpu().numpy(), r["dw2"])
        assert rel < 0.05, f"{mode}: dW2 differs from the oracle's by {rel:.3e}"


@pytest.mark.parametrize("mode", ["high_precision", "dequantized"])
def test_mxfp8_layer_bf16_backward(mode):
    """The same backward modes after an MXFP8 forward: BF16 GEMMs on the BF16
    operands or on the dequantised row-wise MXFP8 copies, against the
    oracle's MXFP8 forward + BF16 backward (GEMM tolerance whole; the MXFP8
    re-quantisation of D keeps the chain within it)."""
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B_BWD, T=400, H=512, I=256, E=6, k=4)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    dy = synth.moe_grad_out(shape, device="cuda")
    layer = MXFP8MoE(T, H, I, E, k)
    layer.quantize_weights(w1, w2)
    layer.forward(x, ids.cuda(), prob.cuda())
    layer.prepare_backward_weights(mode, w1=w1, w2=w2)
    dx, dw1, dw2 = layer.backward_bf16(dy, mode)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    with np.errstate(over="ignore"):
        r = MO.mxfp8_moe_bf16_backward(np_bf16(x).astype(np.float64), ids.numpy(), prob.numpy(),
                                       np_bf16(w1).astype(np.float64), np_bf16(w2).astype(np.float64),
                                       np_bf16(dy).astype(np.float64), E, mode, pad=256)
    R = int(r["seg"][-1])
    _close(np_bf16(layer.c1[:R]), r["c1"], f"MXFP8 {mode}: C")
    _close(np_bf16(layer.dh[:R]), r["dh"], f"MXFP8 {mode}: dH")
    _close(np_bf16(layer.dxp[:R]), r["dxp"], f"MXFP8 {mode}: dX_perm")
    _close(np_bf16(dx), r["dx"], f"MXFP8 {mode}: dX")
    _close(dw1.cpu().numpy(), r["dw1"], f"MXFP8 {mode}: dW1")
    _close(dw2.cpu().numpy(), r["dw2"], f"MXFP8 {mode}: dW2")
