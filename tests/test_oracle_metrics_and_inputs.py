"""Pins for the error metrics and the seeded input generator (CPU only)."""
import math
import os

import numpy as np
import torch

from oracle import metrics as Mx
from microscaled_precision_moe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pairs():
    rows = [l for l in open(os.path.join(GOLDEN, "metrics_pairs.txt")).read().split("\n")
            if l and not l.startswith("#")]
    return [tuple(float(v) for v in r.split(",")) for r in rows[1:]]


def test_snr_rel_l2_identity_reproduces_printed_pair():
    """miniTE report section 2.3: 0.10140 relative L2 <-> 19.88 dB."""
    (snr1, rel1), (snr2, rel2) = _pairs()
    x = np.ones(1000)
    d = np.zeros(1000)
    d[0] = rel1 * math.sqrt(1000)                       # ||d|| / ||x|| = rel1
    assert abs(Mx.rel_l2(x + d, x) - rel1) < 1e-12
    assert round(Mx.snr_db(x + d, x), 2) == snr1
    # the second printed pair is a mean over vectors: Jensen's inequality
    assert snr2 >= -20 * math.log10(rel2)


def test_metric_definitions():
    x = np.array([3.0, 4.0])
    xh = np.array([3.0, 4.5])
    assert Mx.rel_l2(xh, x) == 0.5 / 5.0
    assert abs(Mx.snr_db(xh, x) - 20 * math.log10(10.0)) < 1e-12
    assert Mx.mae(xh, x) == 0.25
    ok, rf, mx, bound = Mx.within_gemm_tolerance(xh, x)
    assert not ok and mx == 0.5 and bound == 0.04


def test_splitmix64_matches_python_reference():
    key = synth.stream_key(0, synth.TID_X)
    idx = torch.tensor([0, 1, 2, 12345, 2 ** 40 + 7], dtype=torch.int64)
    got = synth.words(key, idx)
    for i, g in zip(idx.tolist(), got.tolist()):
        assert (g & ((1 << 64) - 1)) == synth.splitmix64_py(key, i)
    # a published splitmix64 value: state 0 -> first output 0xE220A8397B1DCDAF
    assert synth.splitmix64_py(0, 0) == 0xE220A8397B1DCDAF


def test_generator_distribution_and_slices():
    x = synth.normal_bf16(0, 99, (256, 512)).double()
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    rows = torch.tensor([3, 100, 255])
    part = synth.normal_bf16_rows(0, 99, 512, rows)
    assert torch.equal(part, synth.normal_bf16(0, 99, (256, 512))[rows])
    big = synth.normal_bf16(0, 98, (1 << 20,), outlier_p=1e-3, outlier_mul=50.0).double()
    frac = float((big.abs() > 8).double().mean())
    assert 5e-4 < frac < 1.5e-3


def test_routing_inputs():
    s = synth.scaled(synth.MOE_30B, T=512, E=16)
    ids, pr = synth.routing(s)
    assert ids.shape == (512, 8) and pr.dtype == torch.float32
    assert torch.all((ids >= 0) & (ids < 16))
    assert all(len(set(r.tolist())) == 8 for r in ids)
    assert torch.allclose(pr.sum(1), torch.ones(512), atol=1e-6)
    z = synth.scaled(synth.MOE_671B, T=4096, H=64, I=64, E=256)
    ids, pr = synth.routing(z)
    cnt = torch.bincount(ids.flatten().long(), minlength=256)
    # Zipf(1.1): expert 0 much heavier than the tail
    assert cnt[0] > 10 * cnt[200:].float().mean()
    assert torch.allclose(pr.sum(1), torch.ones(4096), atol=1e-6)


def test_mxfp8_quantizer_input_special_rows():
    x = synth.mxfp8_quantizer_input(M=64, K=64)
    assert x.shape == (160, 64)
    assert torch.all(x[64:96] == 0)
    assert torch.all(x[96:128].abs() == 448)
    sub = x[128:160].view(torch.int16).int() & 0x7FFF
    assert torch.all((sub >= 1) & (sub <= 0x7F))


def test_config5_shape_arithmetic():
    """Post, section "Recipe 2": (61 - 3) * (256 + 1) * 3 * 7168 * 2048 / 1e9
    = 656.5B expert parameters for the DeepSeek-V3-like layer shape."""
    s = synth.MOE_671B
    assert s.H == 7168 and s.I == 2048 and s.E == 256 and s.k == 8
    assert round((61 - 3) * (s.E + 1) * 3 * s.H * s.I / 1e9, 1) == 656.5
