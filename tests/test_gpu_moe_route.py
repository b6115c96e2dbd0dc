"""GPU parity of the expert segment build, gather and combine (integer work:
bit-exact against the oracle)."""
import numpy as np
import pytest
import torch

from oracle import moe as MO
from oracle import quant as Q
from oracle import formats as F
from microscaled_precision_moe_gb300 import synth
from tests.gpu_util import need_gpu, np_bf16, u8, assert_bytes_equal, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _ops():
    from microscaled_precision_moe_gb300 import ops
    return ops


def _check_segments(ids, prob, E, pad=128):
    ops = _ops()
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=pad)
    torch.cuda.synchronize()
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), E, pad)
    assert_bytes_equal(seg.cpu().numpy(), rseg, "seg_offsets")
    R = int(rseg[-1])
    assert R <= cap
    assert_bytes_equal(perm.cpu().numpy()[:R], rperm, "perm")
    assert np.all(perm.cpu().numpy()[R:] == -1)
    assert_bytes_equal(inv.cpu().numpy(), rinv, "inv_perm")
    assert_bytes_equal(rp.cpu().numpy()[:R].view(np.uint32), rrp.view(np.uint32), "row_prob")
    assert ops.get_device_status() == 0
    return seg, perm, inv, rp, cap


@pytest.mark.parametrize("pad", [128, 256])
@pytest.mark.parametrize("shape", [
    synth.scaled(synth.MOE_30B, T=1000, E=16),
    synth.scaled(synth.MOE_671B, T=3000, H=64, I=64),
    synth.MOE_30B,
    synth.MOE_671B,
])
def test_segments_workloads(shape, pad):
    ids, prob = synth.routing(shape)
    _check_segments(ids, prob, shape.E, pad)


def test_segments_edge_cases():
    # one expert takes everything; most experts empty; k = 1; T = 1
    ids = torch.zeros(300, 1, dtype=torch.int32) + 5
    _check_segments(ids, torch.ones(300, 1), 8)
    ids = torch.tensor([[3, 1]], dtype=torch.int32)
    _check_segments(ids, torch.tensor([[0.25, 0.75]]), 4)
    # exactly 128 rows per expert (no padding)
    ids = torch.arange(256, dtype=torch.int32).remainder(2).view(128, 2)
    _check_segments(ids, torch.full((128, 2), 0.5), 2)
    _check_segments(ids, torch.full((128, 2), 0.5), 2, pad=256)


def test_segments_bad_id_sets_device_status():
    ops = _ops()
    ids = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32).cuda()   # 9 >= E
    prob = torch.ones(2, 2).cuda()
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids, prob, 4)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 7          # MPM_ERR_DEVICE_BOUNDS
    assert int(inv[1].item()) == -1
    assert ops.get_device_status() == 0          # reset by the read


@pytest.mark.parametrize("pad", [128, 256])
@pytest.mark.parametrize("T,H,E,k,strided", [(700, 512, 12, 4, False), (300, 7168, 16, 8, True),
                                              (257, 1024, 9, 1, False), (130, 2048, 20, 6, True)])
def test_nvfp4_quantize_scatter_equals_quantize_then_gather(T, H, E, k, strided, pad):
    """The fused quantiser writes the routed rows exactly as the per-token
    quantiser followed by the NVFP4 gather: every byte of the codes, tiled
    scales, token scales and amax slots, padding rows included, and neither
    touches rows at or past the segment end (sentinel bytes stay)."""
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=T, H=H, E=E, k=k)
    ids, prob = synth.routing(shape)
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=pad)
    base = synth.normal_bf16(9, 40 + H, (T, H + (64 if strided else 0)), "cuda", std=2.0,
                             outlier_p=0.01, outlier_mul=50.0)
    x = base[:, :H] if strided else base

    def bufs():
        return ((torch.full((cap, H // 2), 0xA5, dtype=torch.uint8, device="cuda"),
                 torch.full((ops.scale_bytes(cap, H // 16),), 0x5A, dtype=torch.uint8,
                            device="cuda"),
                 torch.full((cap,), 3.0, dtype=torch.float32, device="cuda")),
                torch.full((cap,), 7.0, dtype=torch.float32, device="cuda"))
    got, got_amax = bufs()
    ref, ref_amax = bufs()
    ops.nvfp4_quantize_scatter(x, inv, perm, seg, E, k, cap, out=got, amax_zero=got_amax)
    q, s, ts = ops.nvfp4_quantize_per_token(x)
    ops.moe_gather_nvfp4(q, s, ts, H, perm, seg, E, k, cap, out=ref, amax_zero=ref_amax)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    for g, r, what in zip(got + (got_amax,), ref + (ref_amax,),
                          ("codes", "scales", "token scales", "amax slots")):
        assert torch.equal(g.view(torch.uint8), r.view(torch.uint8)), what
    # the routed rows against the oracle's per-token encoding
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), E, pad)
    R = int(rseg[-1])
    rq, rs, rts = Q.nvfp4_quantize_per_token(np_bf16(x))
    assert_bytes_equal(u8(got[0])[:R], MO.gather_rows(rq, rperm, k), "codes vs oracle")
    got_s = Q.unswizzle_scales(u8(got[1]), cap, H // 16)[:R]
    assert_bytes_equal(got_s, MO.gather_rows(rs, rperm, k), "scales vs oracle")
    assert np.all(u8(got[0])[R:] == 0xA5), "codes written past the segment end"


def test_nvfp4_quantize_scatter_bad_row_sets_status():
    """A routed-row index at or past the segment end is dropped and reported
    (MPM_ERR_DEVICE_BOUNDS); the other rows are still written."""
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=64, H=256, E=4, k=2)
    ids, prob = synth.routing(shape)
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), shape.E)
    x = synth.moe_activations(shape, device="cuda")
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    bad = inv.clone()
    bad[5] = int(seg[-1].item())                  # one past the last valid row
    out = ops.nvfp4_quantize_scatter(x, bad, perm, seg, shape.E, shape.k, cap)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 7
    q, s, ts = ops.nvfp4_quantize_per_token(x)
    row = int(inv[4].item())                        # token 2, slot 0: still written
    assert torch.equal(out[0][row], q[2])


@pytest.mark.parametrize("pad", [128, 256])
@pytest.mark.parametrize("T,H,E,k,strided", [(700, 512, 12, 4, False), (300, 2080, 16, 8, True),
                                              (1000, 2048, 128, 8, False), (500, 256, 10, 6, False),
                                              (200, 64, 3, 1, False)])
def test_mxfp8_quantize_gather_equals_gather_then_quantize(T, H, E, k, strided, pad):
    """The MXFP8 quantiser reading the routed rows straight from the token
    rows writes exactly what the bf16 gather followed by the quantiser (with
    the device row count) writes: every byte of both code copies and both
    scale tiles, sentinel bytes past the segment end included.  H = 2080
    leaves a 32-column last tile; the routed rows against the oracle's
    gather and MXFP8 encoding."""
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=T, H=H, E=E, k=k)
    ids, prob = synth.routing(shape)
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=pad)
    base = synth.normal_bf16(9, 60 + H, (T, H + (64 if strided else 0)), "cuda", std=2.0,
                             outlier_p=0.01, outlier_mul=1e3)
    x = base[:, :H] if strided else base
    ldc = cap + 16

    def bufs():
        return {"row_q": torch.full((cap, H), 0xA5, dtype=torch.uint8, device="cuda"),
                "row_s": torch.full((ops.scale_bytes(cap, H // 32),), 0x5A, dtype=torch.uint8,
                                    device="cuda"),
                "col_q": torch.full((H, ldc), 0xA5, dtype=torch.uint8, device="cuda"),
                "col_s": torch.full((ops.scale_bytes(H, (cap + 31) // 32),), 0x5A,
                                    dtype=torch.uint8, device="cuda")}
    got = ops.mxfp8_quantize_gather(x, perm, seg, E, k, cap, ldc=ldc, out=bufs())
    # the gathered matrix by plain indexing (the library's bf16 gather wants
    # K % 64 == 0), rows past the segment end left as they are
    xp = torch.zeros(cap, H, dtype=torch.bfloat16, device="cuda")
    real = perm >= 0
    xp[real] = x[(perm[real] // k).long()]
    ref = ops.mxfp8_quantize(xp, ldc=ldc, m_valid=seg[E:], out=bufs())
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    for name in ("row_q", "row_s", "col_q", "col_s"):
        assert torch.equal(got[name], ref[name]), name
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), E, pad)
    R = int(rseg[-1])
    xg = MO.gather_rows(np_bf16(x), rperm, k)
    rq, rs = Q.mxfp8_quantize_rowwise(xg)
    assert_bytes_equal(u8(got["row_q"])[:R], rq, "row codes vs oracle")
    assert_bytes_equal(Q.unswizzle_scales(u8(got["row_s"]), cap, H // 32)[:R], rs,
                       "row scales vs oracle")
    cq, cs = Q.mxfp8_quantize_colwise(xg)
    assert_bytes_equal(u8(got["col_q"])[:, :R], cq, "column codes vs oracle")
    assert_bytes_equal(Q.unswizzle_scales(u8(got["col_s"]), H, (cap + 31) // 32)[:, :R // 32],
                       cs, "column scales vs oracle")
    assert np.all(u8(got["row_q"])[R:] == 0xA5), "row codes written past the segment end"
    assert np.all(u8(got["col_q"])[:, R:] == 0xA5), "column codes written past the segment end"


@pytest.mark.parametrize("case", ["one_token", "one_expert", "no_padding", "sparse"])
def test_mxfp8_quantize_gather_degenerate_routings(case):
    """Degenerate routings through the gather form, byte for byte against
    the oracle's gather and MXFP8 encoding: a single token (two rows, each
    its own padded segment), every row on one expert of eight (the other
    segments empty), segments that need no padding (every tile full), and
    most experts empty with a single row on the last one."""
    ops = _ops()
    if case == "one_token":
        ids, prob, E, H = torch.tensor([[3, 1]], dtype=torch.int32), torch.tensor([[0.25, 0.75]]), 4, 64
    elif case == "one_expert":
        ids, prob, E, H = torch.zeros(300, 1, dtype=torch.int32) + 5, torch.ones(300, 1), 8, 320
    elif case == "no_padding":
        ids = torch.arange(512, dtype=torch.int32).remainder(2).view(256, 2)
        prob, E, H = torch.full((256, 2), 0.5), 2, 256
    else:
        ids = torch.zeros(40, 1, dtype=torch.int32)
        ids[-1, 0] = 63
        prob, E, H = torch.ones(40, 1), 64, 128
    T, k = ids.shape
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), E, pad=256)
    x = synth.normal_bf16(4, 11 + H, (T, H), "cuda", std=3.0, outlier_p=0.05, outlier_mul=1e3)
    got = ops.mxfp8_quantize_gather(x, perm, seg, E, k, cap, ldc=cap + 32)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), E, 256)
    R = int(rseg[-1])
    xg = MO.gather_rows(np_bf16(x), rperm, k)
    rq, rs = Q.mxfp8_quantize_rowwise(xg)
    cq, cs = Q.mxfp8_quantize_colwise(xg)
    assert_bytes_equal(u8(got["row_q"])[:R], rq, f"{case}: row codes")
    assert_bytes_equal(Q.unswizzle_scales(u8(got["row_s"]), cap, H // 32)[:R], rs, f"{case}: row scales")
    assert_bytes_equal(u8(got["col_q"])[:, :R], cq, f"{case}: column codes")
    assert_bytes_equal(Q.unswizzle_scales(u8(got["col_s"]), H, (cap + 31) // 32)[:, :R // 32], cs,
                       f"{case}: column scales")


def test_mxfp8_quantize_gather_bad_token_sets_status():
    """A routed row naming a token at or past T reads as zero and is
    reported (MPM_ERR_DEVICE_BOUNDS); the other rows are still quantised."""
    ops = _ops()
    shape = synth.scaled(synth.MOE_30B, T=64, H=256, E=4, k=2)
    ids, prob = synth.routing(shape)
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), shape.E)
    x = synth.moe_activations(shape, device="cuda")
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    bad = perm.clone()
    row = int(inv[6].item())                        # token 3, slot 0
    bad[row] = shape.T * shape.k                    # token T: out of range
    got = ops.mxfp8_quantize_gather(x, bad, seg, shape.E, shape.k, cap)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 7
    ref = ops.mxfp8_quantize(ops.moe_gather_bf16(x, perm, seg, shape.E, shape.k, cap),
                             m_valid=seg[shape.E:])
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    assert torch.all(got["row_q"][row] == 0)
    other = int(inv[8].item())                      # token 4, slot 0
    assert torch.equal(got["row_q"][other], ref["row_q"][other])


def test_gather_bf16_and_nvfp4_and_combine():
    shape = synth.scaled(synth.MOE_30B, T=700, H=512, E=12, k=4)
    ids, prob = synth.routing(shape)
    ops = _ops()
    seg, perm, inv, rp, cap = ops.moe_build_segments(ids.cuda(), prob.cuda(), shape.E)
    x = synth.moe_activations(shape, device="cuda")
    xp = ops.moe_gather_bf16(x, perm, seg, shape.E, shape.k, cap)
    q, s, ts = ops.nvfp4_quantize_per_token(x)
    dq, ds, dts = ops.moe_gather_nvfp4(q, s, ts, shape.H, perm, seg, shape.E, shape.k, cap)
    torch.cuda.synchronize()
    rseg, rperm, rinv, rrp = MO.build_segments(ids.numpy(), prob.numpy(), shape.E)
    R = int(rseg[-1])
    xn = np_bf16(x)
    ref = MO.gather_rows(xn, rperm, shape.k)
    assert np.array_equal(np_bf16(xp)[:R], ref)
    rq, rs, rts = Q.nvfp4_quantize_per_token(xn)
    assert_bytes_equal(u8(dq)[:R], MO.gather_rows(rq, rperm, shape.k), "gathered codes")
    got_s = Q.unswizzle_scales(u8(ds), cap, shape.H // 16)[:R]
    assert_bytes_equal(got_s, MO.gather_rows(rs, rperm, shape.k), "gathered scales")
    assert_bytes_equal(dts.cpu().numpy()[:R].view(np.uint32),
                       MO.gather_rows(rts, rperm, shape.k).view(np.uint32), "gathered ts")
    # combine: y_perm = gathered bf16 rows scaled per row (padding rows are
    # never referenced); the output equals the oracle's combine bit for bit
    y = (xp.float() * torch.linspace(0.5, 1.5, cap, device="cuda")[:, None]).to(torch.bfloat16)
    out = ops.moe_combine(y, inv, shape.T, shape.k)
    torch.cuda.synchronize()
    ref_out = MO.combine(np_bf16(y)[:R], rinv, shape.T, shape.k)
    assert_bytes_equal(bf16_bits(out), F.f64_to_bf16_bits(ref_out), "combine")


def test_combine_cancellation_and_signed_zero():
    """Rows chosen so the binary32 running sum rounds, cancels to zero and
    meets signed zeros: the kernel equals the oracle's combine bit for bit."""
    ops = _ops()
    T, k, H = 64, 8, 256
    rng = np.random.default_rng(7)
    base = rng.standard_normal((T * k, H)) * 2.0 ** rng.integers(-20, 20, (T * k, 1))
    y = torch.from_numpy(base).to(torch.bfloat16)
    yv = y.float().numpy()
    # token 0: x, -x pairs (exact cancellation to +0); token 1: all -0.0
    yv[0:8] = np.repeat(yv[0:1], 8, axis=0) * np.array([1, -1] * 4)[:, None]
    yv[8:16] = -0.0
    # token 2: 1, 2**-8, 2**-30 ... (binary32 loses the tail, bf16 tie to even)
    yv[16:24] = 0.0
    yv[16], yv[17], yv[18] = 1.0, 2.0 ** -8, 2.0 ** -30
    y = torch.from_numpy(yv).to(torch.bfloat16)
    perm_rows = rng.permutation(T * k).astype(np.int32)          # any row order
    y_perm = torch.empty_like(y)
    y_perm[torch.from_numpy(perm_rows.astype(np.int64))] = y
    inv = torch.from_numpy(perm_rows).cuda()
    out = ops.moe_combine(y_perm.cuda(), inv, T, k)
    torch.cuda.synchronize()
    ref = MO.combine(y_perm.float().numpy(), perm_rows, T, k)
    assert_bytes_equal(bf16_bits(out), F.f64_to_bf16_bits(ref), "combine")
    assert np.all(bf16_bits(out[1]) == 0)                        # +0, not -0
