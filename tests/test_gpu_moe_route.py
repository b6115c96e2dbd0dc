"""GPU parity of the expert segment build, gather and combine (integer work:
bit-exact against the oracle)."""
import numpy as np
import pytest
import torch

from oracle import moe as MO
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
    # combine: y_perm = gathered bf16 rows scaled per row; out = slot-order fp32 sum
    y = (xp.float() * torch.linspace(0.5, 1.5, cap, device="cuda")[:, None]).to(torch.bfloat16)
    out = ops.moe_combine(y, inv, shape.T, shape.k)
    torch.cuda.synchronize()
    yn = np_bf16(y).astype(np.float64)
    inv_n = rinv.reshape(shape.T, shape.k)
    acc = np.zeros((shape.T, shape.H), dtype=np.float32)
    for j in range(shape.k):
        acc = (acc + yn[inv_n[:, j]].astype(np.float32)).astype(np.float32)   # fp32, slot order
    ref_out = F.bf16_bits_to_f32(F.f32_to_bf16_bits(acc))
    assert np.array_equal(np_bf16(out), ref_out)
