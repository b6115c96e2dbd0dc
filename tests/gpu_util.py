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


def bf16_bits(t):
    """A bf16 torch tensor -> its uint16 bit patterns (signed zeros kept)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_combine_check(out, y_perm, inv, T, k, what, chunk=4096):
    """The combine kernel's output `out` [T, H] (bf16, on the device) equals,
    bit for bit, the oracle's combine of the kernel's own rows `y_perm`
    under the inverse permutation `inv` [T*k].  The rows are fetched a chunk
    of tokens at a time, so this holds at any size."""
    from oracle import formats as F
    from oracle import moe as MO
    inv = np.asarray(inv, dtype=np.int64).reshape(T, k)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        idx = torch.from_numpy(inv[t0:t1].reshape(-1)).to(y_perm.device)
        rows = y_perm.index_select(0, idx).float().cpu().numpy()
        ref = MO.combine(rows, np.arange(rows.shape[0]), t1 - t0, k)
        got = bf16_bits(out[t0:t1])
        want = F.f64_to_bf16_bits(ref)
        bad = np.flatnonzero(got.ravel() != want.ravel())
        assert bad.size == 0, (f"{what}: {bad.size} of {got.size} outputs differ from the oracle's "
                               f"combine (tokens {t0}..{t1}); first flat {bad[0]}")


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
