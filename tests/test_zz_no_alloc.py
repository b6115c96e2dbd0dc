"""The allocation-free weight quantiser (mpm_nvfp4_quantize_weight_noalloc).

It exists for callers that cannot allocate device memory where they quantise
weights; it keeps its per-expert amax scratch in a fixed device array of the
library instead of a caller-provided workspace.  Its output must equal the
workspace-based mpm_nvfp4_quantize_weight byte for byte, on consecutive calls
(the shared scratch keeps the previous call's contents and must be cleared by
each call).  This file is collected last, and passes on its own in a fresh
process as well as after the rest of the suite.
"""
import ctypes as C

import pytest
import torch

from microscaled_precision_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_moe_gb300 import build, _lib
    build.build()
    return _lib.load()


def _scale_bytes(lib, rows, cols):
    return int(lib.mpm_scale_bytes(rows, cols))


def _outputs(lib, E, R, K):
    return (torch.empty(E, R, K // 2, dtype=torch.uint8, device="cuda"),
            torch.empty(E * _scale_bytes(lib, R, K // 16), dtype=torch.uint8, device="cuda"),
            torch.empty(E, dtype=torch.float32, device="cuda"))


def _quantize_both(lib, parts):
    E, _, K = parts[0].shape
    R = sum(p.shape[1] for p in parts)
    n = len(parts)
    ptrs = (C.c_void_p * n)(*[p.data_ptr() for p in parts])
    rows = (C.c_int64 * n)(*[p.shape[1] for p in parts])
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    # existing entry point, caller-allocated workspace
    ref = _outputs(lib, E, R, K)
    ws = torch.empty(int(lib.mpm_nvfp4_weight_workspace_bytes(E)), dtype=torch.uint8, device="cuda")
    st = lib.mpm_nvfp4_quantize_weight(ptrs, rows, n, K, E, C.c_void_p(ref[0].data_ptr()),
                                       C.c_void_p(ref[1].data_ptr()), C.c_void_p(ref[2].data_ptr()),
                                       C.c_void_p(ws.data_ptr()), ws.numel(), stream)
    assert st == 0
    # allocation-free entry point
    got = _outputs(lib, E, R, K)
    st = lib.mpm_nvfp4_quantize_weight_noalloc(ptrs, rows, n, K, E, C.c_void_p(got[0].data_ptr()),
                                               C.c_void_p(got[1].data_ptr()),
                                               C.c_void_p(got[2].data_ptr()), stream)
    assert st == 0
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_weight_quantiser_matches_workspace_version_twice(lib):
    # first call: large-magnitude weights with outliers, 6 experts, gate + up parts
    big = synth.scaled(synth.MOE_671B, H=512, I=256, E=6)
    w1, _ = synth.moe_weights(big, device="cuda")
    w1 = (w1.float() * 50.0).to(torch.bfloat16)
    parts = [w1[:, :256].contiguous(), w1[:, 256:].contiguous()]
    ref, got = _quantize_both(lib, parts)
    for r, g in zip(ref, got):
        assert torch.equal(r, g)
    # second call right after: smaller weights and fewer experts; a scratch
    # left holding the first call's larger amax would change every byte
    small = synth.scaled(synth.MOE_30B, H=1024, I=128, E=3)
    w1b, w2b = synth.moe_weights(small, device="cuda")
    ref2, got2 = _quantize_both(lib, [w2b.contiguous()])
    for r, g in zip(ref2, got2):
        assert torch.equal(r, g)
    assert float(got2[2].max()) < float(got[2].min())      # the scales really differ


def test_noalloc_rejects_too_many_experts(lib):
    w = torch.zeros(1, 128, 64, dtype=torch.bfloat16, device="cuda")
    ptrs = (C.c_void_p * 1)(w.data_ptr())
    rows = (C.c_int64 * 1)(128)
    dummy = C.c_void_p(w.data_ptr())
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.mpm_nvfp4_quantize_weight_noalloc(ptrs, rows, 1, 64, 4097, dummy, dummy, dummy,
                                                 stream) == 2          # MPM_ERR_SHAPE
