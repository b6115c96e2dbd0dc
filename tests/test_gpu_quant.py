"""GPU parity of the quantisers against the oracle: every code and scale byte
must match (the quantisers are an encoding, so parity is bit-exact)."""
import numpy as np
import pytest
import torch

from oracle import quant as Q
from oracle import formats as F
from microscaled_precision_moe_gb300 import synth
from tests.gpu_util import need_gpu, np_bf16, u8, assert_bytes_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _ops():
    from microscaled_precision_moe_gb300 import ops
    return ops


def _check_nvfp4(x_dev, amax=None, rows=None):
    ops = _ops()
    q, s, ts = ops.nvfp4_quantize_per_token(x_dev, amax_in=amax)
    torch.cuda.synchronize()
    x = np_bf16(x_dev)
    M, K = x.shape
    sel = np.arange(M) if rows is None else np.asarray(rows)
    a_ref = None if amax is None else amax.cpu().numpy()[sel]
    rq, rs, rts = Q.nvfp4_quantize_per_token(x[sel], a_ref)
    assert_bytes_equal(u8(q)[sel], rq, "nvfp4 codes")
    got_s = Q.unswizzle_scales(u8(s), M, K // 16)[sel]
    assert_bytes_equal(got_s, rs, "nvfp4 block scales")
    assert_bytes_equal(ts.cpu().numpy()[sel].view(np.uint32), rts.view(np.uint32), "token scales")
    if rows is None:
        # padding bytes of the last tile are zero
        ref_full = Q.swizzle_scales(rs)
        assert_bytes_equal(u8(s), ref_full, "nvfp4 tiled scale bytes")


def test_nvfp4_single_expert_activation():
    x, _, _ = synth.single_expert_inputs(device="cuda")
    _check_nvfp4(x)


@pytest.mark.parametrize("M,K", [(1, 64), (5, 128), (6, 320), (129, 768), (33, 1024), (2, 1088),
                                 (300, 2048), (77, 7168), (64, 8192)])
def test_nvfp4_shapes(M, K):
    x = synth.normal_bf16(3, 50 + K, (M, K), "cuda", std=2.0, outlier_p=0.01, outlier_mul=100.0)
    _check_nvfp4(x)


def test_nvfp4_strided_input_and_amax_reuse():
    base = synth.normal_bf16(4, 60, (96, 1024 + 64), "cuda")
    x = base[:, :1024]
    amax = x.float().abs().amax(dim=1).contiguous()
    ops = _ops()
    q1, s1, t1 = ops.nvfp4_quantize_per_token(x)
    q2, s2, t2 = ops.nvfp4_quantize_per_token(x, amax_in=amax)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2) and torch.equal(t1, t2)
    _check_nvfp4(x)


def test_nvfp4_extremes():
    K = 256
    rows = []
    rows.append(np.zeros(K))
    rows.append(np.full(K, F.bf16_bits_to_f32(np.array([0x7F7F], np.uint16))[0]))
    rows.append(F.bf16_bits_to_f32(np.arange(1, K + 1, dtype=np.uint16) % 127 + 1))
    neg_small = np.zeros(K)
    neg_small[0] = 6.0
    neg_small[1:] = -0.01
    neg_small[100] = -0.0
    rows.append(neg_small)
    one = np.zeros(K)
    one[40] = -3.0
    rows.append(one)
    ties = np.tile(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25,
                             -1.75, -2.5, -3.5, -5.0, 0.0]), K // 16)
    rows.append(ties)
    x = torch.from_numpy(np.stack(rows).astype(np.float32)).to(torch.bfloat16).cuda()
    _check_nvfp4(x)


def test_nvfp4_activation_large_sample():
    """The 32768 x 7168 activation of the 671B-shaped layer, on sampled rows,
    plus the 16384 x 2048 one in full."""
    s = synth.MOE_671B
    x = synth.moe_activations(s, device="cuda")
    rows = np.random.default_rng(0).choice(s.T, 256, replace=False)
    _check_nvfp4(x, rows=rows)
    del x
    x = synth.moe_activations(synth.MOE_30B, device="cuda")
    _check_nvfp4(x)


def test_nvfp4_weight_joint_scale():
    _, wg, wu = synth.single_expert_inputs(device="cuda")
    ops = _ops()
    q, s, ts = ops.nvfp4_quantize_weight([wg[None].contiguous(), wu[None].contiguous()])
    torch.cuda.synchronize()
    rq, rs, rts = Q.nvfp4_quantize_joint([np_bf16(wg)[None], np_bf16(wu)[None]], 1)
    assert_bytes_equal(u8(q), rq, "weight codes")
    assert_bytes_equal(u8(s), Q.swizzle_scales(rs[0]), "weight scales")
    assert_bytes_equal(ts.cpu().numpy().view(np.uint32), rts.view(np.uint32), "weight s_g")


def test_nvfp4_weight_experts_with_outliers():
    s = synth.scaled(synth.MOE_671B, H=1024, I=256, E=6)
    w1, w2 = synth.moe_weights(s, device="cuda")
    I = s.I
    ops = _ops()
    g, u = w1[:, :I].contiguous(), w1[:, I:].contiguous()
    q, sc, ts = ops.nvfp4_quantize_weight([g, u])
    q2, sc2, ts2 = ops.nvfp4_quantize_weight([w2])
    torch.cuda.synchronize()
    rq, rs, rts = Q.nvfp4_quantize_joint([np_bf16(g), np_bf16(u)], s.E)
    assert_bytes_equal(u8(q), rq, "W1 codes")
    per = Q.scale_bytes(2 * I, s.H // 16)
    for e in range(s.E):
        assert_bytes_equal(u8(sc)[e * per:(e + 1) * per], Q.swizzle_scales(rs[e]), f"W1 scales e{e}")
    assert_bytes_equal(ts.cpu().numpy().view(np.uint32), rts.view(np.uint32), "W1 s_g")
    rq2, rs2, rts2 = Q.nvfp4_quantize_joint([np_bf16(w2)], s.E)
    assert_bytes_equal(u8(q2), rq2, "W2 codes")
    assert_bytes_equal(ts2.cpu().numpy().view(np.uint32), rts2.view(np.uint32), "W2 s_g")


@pytest.mark.parametrize("E,R,K,parts", [
    (2, 4096, 7168, 1),     # two 671B-shaped W1 experts, the widest rows
    (40, 128, 64, 2),       # many small experts, the narrowest rows
    (9, 384, 2048, 3),      # three parts of 128 rows sharing one scale
])
def test_nvfp4_weight_shapes(E, R, K, parts):
    """The joint weight quantiser (per-expert amax pass, then the encode):
    every code, scale byte and outer scale against the oracle's joint
    quantisation, from the widest to the narrowest rows and with up to
    three parts per expert."""
    ops = _ops()
    w = synth.normal_bf16(3, 40 + E, (E, R, K), "cuda", std=0.01, outlier_p=1e-4,
                          outlier_mul=100.0)
    w[E // 2] *= 1e-3                                  # one expert on another scale
    rp = R // parts
    pieces = [w[:, i * rp:(i + 1) * rp].contiguous() for i in range(parts)]
    q, sc, ts = ops.nvfp4_quantize_weight(pieces)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    rq, rs, rts = Q.nvfp4_quantize_joint([np_bf16(p) for p in pieces], E)
    assert_bytes_equal(u8(q), rq, "codes")
    per = Q.scale_bytes(R, K // 16)
    for e in range(E):
        assert_bytes_equal(u8(sc)[e * per:(e + 1) * per], Q.swizzle_scales(rs[e]), f"scales e{e}")
    assert_bytes_equal(ts.cpu().numpy().view(np.uint32), rts.view(np.uint32), "s_g")


def _check_mxfp8(x_dev, ldc=None):
    ops = _ops()
    o = ops.mxfp8_quantize(x_dev, ldc=ldc)
    torch.cuda.synchronize()
    x = np_bf16(x_dev)
    M, K = x.shape
    rq, rs = Q.mxfp8_quantize_rowwise(x)
    assert_bytes_equal(u8(o["row_q"]), rq, "mxfp8 row codes")
    assert_bytes_equal(u8(o["row_s"]), Q.swizzle_scales(rs), "mxfp8 row scales (tiled, padded)")
    cq, cs = Q.mxfp8_quantize_colwise(x)
    assert_bytes_equal(u8(o["col_q"])[:, :M], cq, "mxfp8 col codes")
    assert_bytes_equal(u8(o["col_s"]), Q.swizzle_scales(cs), "mxfp8 col scales (tiled, padded)")


def test_mxfp8_quantizer_workload():
    """8192 x 2048 activations (1% rows x1e3) plus 32 zero rows, 32 rows of
    +-448 and 32 rows of bf16 subnormals: both copies byte-exact."""
    x = synth.mxfp8_quantizer_input(device="cuda")
    assert x.shape == (8288, 2048)
    _check_mxfp8(x)


def test_mxfp8_bench_size_sampled():
    """The 65536 x 2048 input the benchmark times (about 36 tiles per CTA of
    the persistent grid): row-wise codes and scales of 1024 sampled rows and
    the column-wise codes and scales of 32 sampled 32-row blocks, all
    columns, byte for byte against the oracle."""
    ops = _ops()
    M, K = 65536, 2048
    x_dev = synth.normal_bf16(0, synth.TID_X, (M, K), "cuda")
    o = ops.mxfp8_quantize(x_dev)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    rows = np.sort(np.concatenate([np.arange(128), rng.choice(M, 768, replace=False),
                                   np.arange(M - 128, M)]))
    rows = np.unique(rows)
    xr = np_bf16(x_dev[torch.from_numpy(rows).cuda()])
    rq, rs = Q.mxfp8_quantize_rowwise(xr)
    assert_bytes_equal(u8(o["row_q"])[rows], rq, "row codes (sampled rows)")
    got_rs = Q.unswizzle_scales(u8(o["row_s"]), M, K // 32)[rows]
    assert_bytes_equal(got_rs, rs, "row scales (sampled rows)")
    blocks = np.unique(np.concatenate([[0, M // 32 - 1], rng.choice(M // 32, 30, replace=False)]))
    got_cq = u8(o["col_q"])
    got_cs = Q.unswizzle_scales(u8(o["col_s"]), K, M // 32)
    for b in blocks:
        xb = np_bf16(x_dev[b * 32:(b + 1) * 32])
        cq, cs = Q.mxfp8_quantize_colwise(xb)
        assert_bytes_equal(got_cq[:, b * 32:(b + 1) * 32], cq, f"column codes, block {b}")
        assert_bytes_equal(got_cs[:, b:b + 1], cs, f"column scales, block {b}")


@pytest.mark.parametrize("M,K", [(1, 32), (33, 64), (40, 96), (200, 160), (257, 2048)])
def test_mxfp8_shapes(M, K):
    x = synth.normal_bf16(5, 70 + K, (M, K), "cuda", std=3.0, outlier_p=0.02, outlier_mul=1e4)
    _check_mxfp8(x, ldc=((M + 15) // 16) * 16)


@pytest.mark.parametrize("rowwise,colwise", [(True, True), (True, False), (False, True)])
def test_mxfp8_full_and_edge_tiles_mixed(rowwise, colwise):
    """1000 x 2080: seven full 128 x 64 tiles per column of tiles and a
    ragged eighth, and a 32-column last tile column, so every CTA meets full
    tiles (codes staged in shared memory and stored by TMA) and edge tiles
    (stored per thread) in changing order; then the same input with a
    device row count of 700 and a padded column pitch: rows at and past it
    keep the sentinel bytes."""
    ops = _ops()
    M, K = 1000, 2080
    x_dev = synth.normal_bf16(7, 91, (M, K), "cuda", std=2.0, outlier_p=0.01, outlier_mul=1e3)
    x = np_bf16(x_dev)
    rq, rs = Q.mxfp8_quantize_rowwise(x)
    cq, cs = Q.mxfp8_quantize_colwise(x)
    o = ops.mxfp8_quantize(x_dev, rowwise=rowwise, colwise=colwise)
    torch.cuda.synchronize()
    if rowwise:
        assert_bytes_equal(u8(o["row_q"]), rq, "row codes")
        assert_bytes_equal(u8(o["row_s"]), Q.swizzle_scales(rs), "row scales")
    if colwise:
        assert_bytes_equal(u8(o["col_q"])[:, :M], cq, "col codes")
        assert_bytes_equal(u8(o["col_s"]), Q.swizzle_scales(cs), "col scales")
    mv, ldc = 700, 1024
    out = {}
    if rowwise:
        out["row_q"] = torch.full((M, K), 0xA5, dtype=torch.uint8, device="cuda")
    if colwise:
        out["col_q"] = torch.full((K, ldc), 0xA5, dtype=torch.uint8, device="cuda")
    o = ops.mxfp8_quantize(x_dev, rowwise=rowwise, colwise=colwise, ldc=ldc,
                           m_valid=torch.tensor([mv], dtype=torch.int32, device="cuda"), out=out)
    torch.cuda.synchronize()
    xv = x.copy()
    xv[mv:] = 0
    if rowwise:
        got = u8(o["row_q"])
        assert_bytes_equal(got[:mv], Q.mxfp8_quantize_rowwise(xv[:mv])[0], "row codes, m_valid")
        assert (got[mv:] == 0xA5).all(), "row codes written past m_valid"
    if colwise:
        got = u8(o["col_q"])
        assert_bytes_equal(got[:, :mv], Q.mxfp8_quantize_colwise(xv)[0][:, :mv], "col codes, m_valid")
        assert (got[:, mv:] == 0xA5).all(), "col codes written past m_valid"


def test_mxfp8_reads_what_the_previous_kernel_wrote():
    """The MXFP8 quantiser is launched as a programmatic dependent of the
    kernel before it in the stream.  Here that kernel is a long matmul whose
    result is the quantiser's input, and the quantiser's output buffers were
    read by the kernel before that: with no host synchronisation in
    between, the codes must still be those of the matmul's result."""
    ops = _ops()
    M, K = 2048, 4096
    a = synth.normal_bf16(8, 1, (M, 4096), "cuda")
    b = synth.normal_bf16(8, 2, (4096, K), "cuda", std=0.02)
    x = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    o = ops.mxfp8_quantize(torch.zeros(M, K, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for _ in range(3):
        probe = o["row_q"].float().sum() + o["col_q"].float().sum()   # reads the outputs
        torch.matmul(a, b, out=x)                                        # writes the input
        ops.mxfp8_quantize(x, out=o)
    torch.cuda.synchronize()
    assert probe.item() >= 0
    xn = np_bf16(x)
    rq, rs = Q.mxfp8_quantize_rowwise(xn)
    cq, cs = Q.mxfp8_quantize_colwise(xn)
    assert_bytes_equal(u8(o["row_q"]), rq, "row codes after a producing matmul")
    assert_bytes_equal(u8(o["col_q"])[:, :M], cq, "col codes after a producing matmul")


def test_quantizers_deterministic():
    x = synth.normal_bf16(6, 80, (512, 2048), "cuda")
    ops = _ops()
    a = ops.nvfp4_quantize_per_token(x)
    b = ops.nvfp4_quantize_per_token(x)
    m1 = ops.mxfp8_quantize(x)
    m2 = ops.mxfp8_quantize(x)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    for k in m1:
        assert torch.equal(m1[k], m2[k])


def test_batch_independence_on_gpu():
    x = synth.normal_bf16(7, 81, (256, 512), "cuda", std=1.0, outlier_p=0.01, outlier_mul=1e3)
    perm = torch.randperm(256, generator=torch.Generator().manual_seed(0)).cuda()
    ops = _ops()
    q, s, ts = ops.nvfp4_quantize_per_token(x)
    qp, sp, tsp = ops.nvfp4_quantize_per_token(x[perm].contiguous())
    q1, s1, ts1 = ops.nvfp4_quantize_per_token(x[17:18].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(q[perm], qp) and torch.equal(ts[perm], tsp)
    assert torch.equal(q[17], q1[0]) and torch.equal(ts[17], ts1[0])
    S = Q.unswizzle_scales(u8(s), 256, 32)
    Sp = Q.unswizzle_scales(u8(sp), 256, 32)
    assert np.array_equal(S[perm.cpu().numpy()], Sp)
