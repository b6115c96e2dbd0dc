"""GPU parity of the single-pass FC2 with online amax compensation ("miniTE
technical report", section 5.6) against the oracle's
``nvfp4_fc2_online_amax`` on identical D:

* the tile-by-tile quantisation (codes, block scales and the outer scale of
  every 256-column tile, against the running row amax): byte-exact;
* the compensated FC2 output Y: the GEMM tolerance;
* the layer output: the oracle's combine of the kernel's own Y, bit for bit.
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
TILE = 256


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _close(got, ref, what):
    ok, rf, mx, bound = Mx.within_gemm_tolerance(got, ref, REL, ELEM)
    assert ok, f"{what}: rel_frob={rf:.3e} max_err={mx:.3e} bound={bound:.3e}"


def _check_online_quant(d_dev, q, s, gs, rows, what):
    """Codes, tiled block scales and per-tile outer scales of rows `rows` of
    D (device bf16) against the oracle's tile-by-tile encoding."""
    dn = np_bf16(d_dev[torch.from_numpy(rows).cuda()])
    I = dn.shape[1]
    w_dummy = Q.nvfp4_quantize_joint([np.zeros((1, 128, I), dtype=np.float32)], 1)
    r = MO.nvfp4_fc2_online_amax(dn, np.array([0, dn.shape[0]]), w_dummy, TILE)
    assert_bytes_equal(u8(q)[rows], Q.pack_e2m1(r["codes"]), f"{what}: codes")
    got_s = Q.unswizzle_scales(u8(s), q.shape[0], I // 16)[rows]
    assert_bytes_equal(got_s, r["sb"], f"{what}: block scales")
    assert_bytes_equal(gs.cpu().numpy()[rows].view(np.uint32), r["gs"].view(np.uint32),
                       f"{what}: tile outer scales")


@pytest.mark.parametrize("I", [256, 768, 2048])
def test_online_quantiser_structured_rows(I):
    """Rows built so the running amax moves in every way the section allows:
    growing from tile to tile, set by the first tile, leading all-zero tiles,
    all-zero rows, a late outlier, subnormal-sized rows; plus random rows."""
    from microscaled_precision_moe_gb300 import ops
    n_t = I // TILE
    M = 384
    base = np.random.default_rng(11).standard_normal((M, I)) * 0.05
    for r in range(64):                                   # amax grows tile by tile
        base[r] *= np.repeat(2.0 ** np.arange(n_t), TILE)
    base[64:96, :TILE] *= 100.0                           # first tile sets the amax
    base[96:128, : TILE * (n_t // 2)] = 0.0              # leading zero tiles
    base[128:144] = 0.0                                   # all-zero rows
    base[144:176, -7] = 1e3                               # a late outlier
    base[176:192] *= 1e-36                                # tiny rows (outer-scale floor)
    x = torch.from_numpy(base).to(torch.bfloat16).cuda()
    q, s, gs = ops.nvfp4_quantize_online(x)
    torch.cuda.synchronize()
    assert gs.shape == (M, n_t)
    _check_online_quant(x, q, s, gs, np.arange(M), f"I={I}")
    # a row's encoding does not depend on the batch around it
    q1, s1, gs1 = ops.nvfp4_quantize_online(x[70:71].contiguous())
    assert torch.equal(q1[0], q[70]) and torch.equal(gs1[0], gs[70])


def _online_layer(shape):
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    layer = NVFP4MoE(shape.T, shape.H, shape.I, shape.E, shape.k, fc2="online")
    out = layer.forward(x, ids.cuda(), prob.cuda(), W)
    torch.cuda.synchronize()
    from microscaled_precision_moe_gb300 import ops
    assert ops.get_device_status() == 0
    return layer, out, W, w2


def _check_expert(layer, W, w2, seg, perm, e, what):
    """One expert's rows: online quantisation bytes and Y against the oracle
    on the kernel's own D (identical operands), W2 quantised by the oracle."""
    r0, r1 = int(seg[e]), int(seg[e + 1])
    rows = np.arange(r0, r1)
    real = rows[perm[r0:r1] >= 0]
    dq, ds, dgs = layer.dq
    _check_online_quant(layer.d, dq, ds, dgs, real, f"{what} expert {e}")
    dn = np_bf16(layer.d[torch.from_numpy(real).cuda()])
    w2q = Q.nvfp4_quantize_joint([np_bf16(w2[e])[None]], 1)
    ref = MO.nvfp4_fc2_online_amax(dn, np.array([0, dn.shape[0]]), w2q, TILE)
    y = np_bf16(layer.y[torch.from_numpy(real).cuda()])
    _close(y, ref["y"], f"{what} expert {e}: online FC2 Y")


def test_online_layer_reduced():
    """A reduced 30B-shaped layer (segments padded to 256 rows, empty and
    ragged experts included): every expert checked, and the combine."""
    shape = synth.scaled(synth.MOE_30B, T=700, H=512, I=768, E=12, k=4)
    layer, out, W, w2 = _online_layer(shape)
    seg, perm, inv, rp = [t.cpu().numpy() for t in layer.seg]
    for e in range(shape.E):
        if seg[e + 1] > seg[e]:
            _check_expert(layer, W, w2, seg, perm, e, "reduced")
    oracle_combine_check(out, layer.y, inv, shape.T, shape.k, "online combine")


def test_online_layer_against_oracle_single_pass():
    """The whole single-pass layer of the oracle (its own quantised X, FC1,
    SwiGLU, online FC2, combine) against the kernel's: the GPU's D differs
    from the oracle's only where fp32 accumulation moves a bf16 rounding, so
    the output meets the chained bound of the two-pass layer."""
    shape = synth.scaled(synth.MOE_30B, T=300, H=512, I=512, E=6, k=4)
    layer, out, W, w2 = _online_layer(shape)
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2c = synth.moe_weights(shape, device="cuda")
    with np.errstate(over="ignore"):
        r = MO.nvfp4_moe_forward_single_pass(np_bf16(x), ids.numpy(), prob.numpy(), np_bf16(w1),
                                             np_bf16(w2c), shape.E, tile_k=TILE, pad=256)
    R = int(r["two_pass"]["seg"][-1])
    d_same = (np_bf16(layer.d)[:R] == r["two_pass"]["d"]).all(axis=1)
    _close(np_bf16(layer.y)[:R][d_same], r["y"][d_same], "online Y on identical D rows")
    rel = Mx.rel_frobenius(np_bf16(out), r["out"])
    print(f"PARITY-STATS online layer: D rows differing {1 - d_same.mean():.4f}, layer rel {rel:.3e}")
    assert rel < 5e-3


def test_online_layer_671b_full_size():
    """The headline workload (32768 tokens, hidden 7168, 256 experts,
    intermediate 2048, Zipf load) with the online FC2: the heaviest, the
    lightest and a middle expert checked whole, the combine whole."""
    shape = synth.MOE_671B
    layer, out, W, w2 = _online_layer(shape)
    seg, perm, inv, rp = [t.cpu().numpy() for t in layer.seg]
    sizes = np.diff(seg)
    nz = np.flatnonzero(sizes > 0)
    order = nz[np.argsort(sizes[nz], kind="stable")]
    for e in (int(order[-1]), int(order[0]), int(order[len(order) // 2])):
        _check_expert(layer, W, w2, seg, perm, e, "671B")
    oracle_combine_check(out, layer.y, inv, shape.T, shape.k, "online combine")
