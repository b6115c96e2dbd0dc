"""Helpers shared by the GPU tests (test infrastructure)."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_moe_gb300 import build
    build.build()


def np_bf16(t):
    """A bf16 torch tensor -> float32 numpy array with the same values."""
    return t.detach().cpu().float().numpy()


def u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def assert_bytes_equal(got, ref, what):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    bad = np.flatnonzero(got.ravel() != ref.ravel())
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {got.size} bytes differ; first at flat "
                             f"{i}: got {got.ravel()[i]} ref {ref.ravel()[i]}")
