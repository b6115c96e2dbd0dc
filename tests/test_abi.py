"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/mpm.h declares, and rejects bad arguments on the host before any
launch (CPU only: none of these calls reaches the GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mpm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(mpm_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from microscaled_precision_moe_gb300 import build, _lib
    build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    from microscaled_precision_moe_gb300 import _lib
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.EXPORTED)


def test_pure_host_queries(lib):
    assert lib.mpm_version() == 101
    assert lib.mpm_scale_bytes(8288, 64) == 8320 * 64
    assert lib.mpm_scale_bytes(2048, 259) == 2048 * 260
    assert lib.mpm_moe_row_capacity(32768, 8, 256, 128) == 262144 + 128 * 256
    assert lib.mpm_moe_row_capacity(32768, 8, 256, 256) == 262144 + 256 * 256
    assert lib.mpm_moe_row_capacity(32768, 8, 256, 64) == 262144 + 64 * 256
    assert lib.mpm_moe_row_capacity(64, 8, 256, 16) == 512 + 16 * 256
    assert lib.mpm_moe_row_capacity(32768, 8, 256, 96) == 0
    assert lib.mpm_status_string(7) == b"MPM_ERR_DEVICE_BOUNDS"


def test_host_validation_rejects_before_launch(lib):
    from microscaled_precision_moe_gb300 import _lib as L
    fake = C.c_void_p(0x10000)          # never dereferenced: validation fails first
    odd = C.c_void_p(0x10008)
    # NULL input
    assert lib.mpm_nvfp4_quantize_per_token(None, 4, 64, 64, None, fake, fake, fake, None, None) == 1
    # K not a multiple of 64 / too large
    assert lib.mpm_nvfp4_quantize_per_token(fake, 4, 48, 64, None, fake, fake, fake, None, None) == 2
    assert lib.mpm_nvfp4_quantize_per_token(fake, 4, 16384, 16384, None, fake, fake, fake, None, None) == 2
    # misaligned input / leading dimension
    assert lib.mpm_nvfp4_quantize_per_token(odd, 4, 64, 64, None, fake, fake, fake, None, None) == 3
    assert lib.mpm_nvfp4_quantize_per_token(fake, 4, 64, 68, None, fake, fake, fake, None, None) == 3
    # MXFP8: no copy requested, K % 32, ldc < M
    assert lib.mpm_mxfp8_quantize(fake, 4, 64, 64, 0, fake, fake, fake, 16, fake, None, None) == 2
    assert lib.mpm_mxfp8_quantize(fake, 4, 40, 40, 1, fake, fake, None, 0, None, None, None) == 2
    assert lib.mpm_mxfp8_quantize(fake, 64, 64, 64, 2, None, None, fake, 32, fake, None, None) == 2
    # segments: E too large, workspace too small
    assert lib.mpm_moe_build_segments(fake, fake, 4, 2, 2048, 128, fake, fake, fake, fake, fake, 1 << 20, None) == 2
    assert lib.mpm_moe_build_segments(fake, fake, 4, 2, 8, 128, fake, fake, fake, fake, fake, 0, None) == 2
    assert lib.mpm_moe_build_segments(fake, fake, 4, 2, 8, 100, fake, fake, fake, fake, fake, 1 << 20, None) == 2
    # GEMM descriptor: bad N, bad K, wgrad on NVFP4
    d = L.GroupedGemmDesc()
    d.kind, d.group, d.epilogue, d.E, d.a_rows, d.N, d.K = 0, 0, 0, 1, 128, 200, 256
    for f in ("a_dev", "b_dev", "sfa_dev", "sfb_dev", "out_dev"):
        setattr(d, f, 0x10000)
    d.lda_bytes = d.ldb_bytes = 128
    d.a_total_rows = d.b_total_rows = 128
    d.sfa_cols = d.sfb_cols = 16
    d.ldo = 256
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 2
    d.N, d.K = 256, 100
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 2
    d.K, d.group = 256, 1
    d.seg_dev = 0x10000
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    d.group, d.tile_m = 0, 192                      # only 128 or 256
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    assert lib.mpm_moe_grouped_gemm(None, None) == 1


def _gemm_desc(kind, group, epi, N, K, tile_m):
    from microscaled_precision_moe_gb300 import _lib as L
    d = L.GroupedGemmDesc()
    d.kind, d.group, d.epilogue, d.tile_m = kind, group, epi, tile_m
    d.E, d.a_rows, d.N, d.K = 1, 256, N, K
    for f in ("a_dev", "b_dev", "out_dev"):
        setattr(d, f, 0x10000)
    d.lda_bytes = d.ldb_bytes = 4096
    d.a_total_rows = d.b_total_rows = 256
    d.ldo = 2 * N
    return d


def test_online_quantiser_and_fc2_validation(lib):
    """The running-amax quantiser and the online FC2 epilogue reject bad
    arguments on the host (CPU only)."""
    from microscaled_precision_moe_gb300 import _lib as L
    fake = C.c_void_p(0x10000)
    odd = C.c_void_p(0x10008)
    assert lib.mpm_nvfp4_quantize_online(None, 4, 256, 256, fake, fake, fake, None, None) == 1
    assert lib.mpm_nvfp4_quantize_online(fake, 4, 320, 320, fake, fake, fake, None, None) == 2
    assert lib.mpm_nvfp4_quantize_online(fake, 0, 256, 256, fake, fake, fake, None, None) == 2
    assert lib.mpm_nvfp4_quantize_online(fake, 4, 256, 128, fake, fake, fake, None, None) == 2
    assert lib.mpm_nvfp4_quantize_online(odd, 4, 256, 256, fake, fake, fake, None, None) == 3
    d = _gemm_desc(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16_ONLINE, 256, 512, 256)
    d.sfa_dev = d.sfb_dev = 0x10000
    d.sfa_cols = d.sfb_cols = 32
    d.seg_dev = 0x10000
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 1          # no tile scales (aux)
    d.aux_dev, d.ld_aux = 0x10000, 2
    d.alpha_a_dev = 0x10000
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4          # per-row scale given
    d.alpha_a_dev = None
    d.ld_aux = 1
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 2          # ld_aux < K / 256
    d.ld_aux = 2
    d.kind = L.KIND_MXFP8
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4          # NVFP4 only
    d.kind, d.tile_m = L.KIND_NVFP4, 128
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4          # CTA pairs only


def test_bf16_mn_major_and_small_m_validation(lib):
    """The BF16 kind, its MN-major operands and the small-M tile mode are
    checked on the host (CPU only)."""
    from microscaled_precision_moe_gb300 import _lib as L
    # BF16 needs the CTA-pair kernel
    d = _gemm_desc(L.KIND_BF16, L.GROUP_M, L.EPI_BF16, 256, 512, 128)
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    # BF16: K % 64
    d = _gemm_desc(L.KIND_BF16, L.GROUP_M, L.EPI_BF16, 256, 96, 256)
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 2
    # MN-major A only in GROUP_K, and only for the bf16 kind
    d = _gemm_desc(L.KIND_BF16, L.GROUP_M, L.EPI_BF16, 256, 512, 256)
    d.a_mn_major = 1
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    d = _gemm_desc(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, 256, 512, 256)
    d.b_mn_major = 1
    d.sfa_dev = d.sfb_dev = 0x10000
    d.sfa_cols = d.sfb_cols = 16
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    # GROUP_K with only one operand MN-major is not a supported combination
    d = _gemm_desc(L.KIND_BF16, L.GROUP_K, L.EPI_F32, 256, 0, 256)
    d.seg_dev = 0x10000
    d.a_mn_major = 1
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    # small-M kernel: GROUP_M only, no bf16, no SwiGLU-save / DSwiGLU
    d = _gemm_desc(L.KIND_BF16, L.GROUP_M, L.EPI_BF16, 256, 512, L.TILE_SMALL_M)
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4
    d = _gemm_desc(L.KIND_NVFP4, L.GROUP_M, L.EPI_DSWIGLU, 256, 512, L.TILE_SMALL_M)
    d.sfa_dev = d.sfb_dev = 0x10000
    d.sfa_cols = d.sfb_cols = 32
    assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == 4


def test_dequantize_and_transpose_validation(lib):
    fake = C.c_void_p(0x10000)
    odd = C.c_void_p(0x10008)
    # NVFP4 -> bf16: NULL, K % 64, rows_per_outer, ldo, alignment
    assert lib.mpm_nvfp4_dequantize(None, fake, fake, 1, 4, 64, fake, 64, None, None) == 1
    assert lib.mpm_nvfp4_dequantize(fake, fake, fake, 1, 4, 48, fake, 64, None, None) == 2
    assert lib.mpm_nvfp4_dequantize(fake, fake, fake, 0, 4, 64, fake, 64, None, None) == 2
    assert lib.mpm_nvfp4_dequantize(fake, fake, fake, 1, 4, 64, fake, 60, None, None) == 2
    assert lib.mpm_nvfp4_dequantize(odd, fake, fake, 1, 4, 64, fake, 64, None, None) == 3
    # MXFP8 -> bf16: K % 32, ldo % 8
    assert lib.mpm_mxfp8_dequantize(fake, fake, 4, 48, fake, 48, None, None) == 2
    assert lib.mpm_mxfp8_dequantize(fake, fake, 4, 64, fake, 68, None, None) == 2
    # transpose: shapes and leading dimensions
    assert lib.mpm_transpose_bf16(None, 4, 4, 4, fake, 4, None, None) == 1
    assert lib.mpm_transpose_bf16(fake, 0, 4, 4, fake, 4, None, None) == 2
    assert lib.mpm_transpose_bf16(fake, 8, 4, 3, fake, 8, None, None) == 2
    assert lib.mpm_transpose_bf16(fake, 8, 4, 4, fake, 7, None, None) == 2


def test_empty_inputs_and_size_limits_are_shape_errors(lib):
    """An empty input (no rows, tokens or experts) and every documented size
    limit return MPM_ERR_SHAPE from the host checks, for every entry point
    that takes sizes (CPU only: none of these calls reaches the GPU)."""
    from microscaled_precision_moe_gb300 import _lib as L
    fake = C.c_void_p(0x10000)
    SHAPE = 2
    # quantisers: no rows
    assert lib.mpm_mxfp8_quantize(fake, 0, 64, 64, 3, fake, fake, fake, 16, fake, None, None) == SHAPE
    assert lib.mpm_nvfp4_quantize_per_token(fake, 0, 64, 64, None, fake, fake, fake, None, None) == SHAPE
    # NVFP4 rows longer than 8192 elements, and ldx < K
    assert lib.mpm_nvfp4_quantize_per_token(fake, 4, 8256, 8256, None, fake, fake, fake, None, None) == SHAPE
    assert lib.mpm_nvfp4_quantize_per_token(fake, 4, 128, 64, None, fake, fake, fake, None, None) == SHAPE
    # joint weight quantiser: no experts, an empty part, R % 128, K > 8192,
    # too many parts, a workspace smaller than the query returns
    parts = (C.c_void_p * 2)(0x10000, 0x20000)

    def wq(rows, nparts=2, K=256, E=4, ws=1 << 16):
        r = (C.c_int64 * 2)(*rows)
        return lib.mpm_nvfp4_quantize_weight(parts, r, nparts, K, E, fake, fake, fake, fake, ws, None)

    assert lib.mpm_nvfp4_weight_workspace_bytes(0) == 0
    assert wq((64, 64), E=0) == SHAPE
    assert wq((0, 128)) == SHAPE
    assert wq((64, 32)) == SHAPE
    assert wq((64, 64), K=8256) == SHAPE
    assert wq((64, 64), nparts=5) == SHAPE
    assert wq((64, 64), ws=lib.mpm_nvfp4_weight_workspace_bytes(4) - 1) == SHAPE
    # segments: no tokens, k out of 1..64, T * k above 2^30
    ws = 1 << 30
    assert lib.mpm_moe_segments_workspace_bytes(0, 8, 16) == 0
    assert lib.mpm_moe_row_capacity(0, 8, 16, 128) == 0
    assert lib.mpm_moe_build_segments(fake, fake, 0, 8, 16, 128, fake, fake, fake, fake, fake, ws, None) == SHAPE
    assert lib.mpm_moe_build_segments(fake, fake, 4, 0, 16, 128, fake, fake, fake, fake, fake, ws, None) == SHAPE
    assert lib.mpm_moe_build_segments(fake, fake, 4, 65, 16, 128, fake, fake, fake, fake, fake, ws, None) == SHAPE
    assert lib.mpm_moe_build_segments(fake, fake, 1 << 28, 8, 16, 128, fake, fake, fake, fake, fake, ws,
                                      None) == SHAPE
    # gather: no tokens, no capacity, K % 64; an unknown kind is unsupported
    g = lambda what, T, K, cap: lib.mpm_moe_gather(what, fake, fake, fake, T, K, 8, fake, fake, 16, cap,
                                                   fake, fake, fake, None, None)
    assert g(L.GATHER_BF16, 0, 256, 1024) == SHAPE
    assert g(L.GATHER_BF16, 4, 256, 0) == SHAPE
    assert g(L.GATHER_NVFP4, 4, 96, 1024) == SHAPE
    assert g(2, 4, 256, 1024) == 4
    # combine: no tokens, H below 8 or not a multiple of 8
    assert lib.mpm_moe_combine(fake, fake, 0, 8, 256, fake, None) == SHAPE
    assert lib.mpm_moe_combine(fake, fake, 4, 8, 4, fake, None) == SHAPE
    assert lib.mpm_moe_combine(fake, fake, 4, 8, 12, fake, None) == SHAPE
    # dequantisation and transpose: no rows / no columns
    assert lib.mpm_nvfp4_dequantize(fake, fake, fake, 1, 0, 64, fake, 64, None, None) == SHAPE
    assert lib.mpm_mxfp8_dequantize(fake, fake, 0, 64, fake, 64, None, None) == SHAPE
    assert lib.mpm_transpose_bf16(fake, 4, 0, 4, fake, 4, None, None) == SHAPE
    # grouped GEMM: no experts, no rows, no operand rows
    for field, value in (("E", 0), ("a_rows", 0), ("a_total_rows", 0), ("b_total_rows", 0)):
        d = _gemm_desc(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, 256, 512, 256)
        d.sfa_dev = d.sfb_dev = 0x10000
        d.sfa_cols = d.sfb_cols = 16
        d.seg_dev = 0x10000
        setattr(d, field, value)
        assert lib.mpm_moe_grouped_gemm(C.byref(d), None) == SHAPE, field


def test_plain_c_client(lib, tmp_path):
    """tests/abi_client.c, compiled as C99 with gcc against include/mpm.h and
    linked with libmpm.so, runs its host-only checks (no GPU, no Python in
    the client)."""
    import shutil
    import subprocess
    from microscaled_precision_moe_gb300 import _lib
    gcc = shutil.which("gcc")
    nvcc = shutil.which("nvcc")
    if gcc is None or nvcc is None:
        pytest.skip("gcc and the CUDA toolkit headers are needed")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path / "abi_client")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "abi_client.c"),
                    "-L", libdir, "-lmpm", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "abi_client: ok" in r.stdout


def test_binding_checks_arguments_before_the_library(lib):
    """The Python binding rejects what the C side cannot see (element type,
    rank, dense rows, buffer sizes) with TypeError / ValueError, and CPU
    tensors with ValueError; nothing here reaches the library's launches."""
    import torch
    from microscaled_precision_moe_gb300 import ops
    bf, i32, f32, u8 = torch.bfloat16, torch.int32, torch.float32, torch.uint8
    x = torch.zeros(8, 64, dtype=bf)
    with pytest.raises(TypeError):
        ops.nvfp4_quantize_per_token(x.float())
    with pytest.raises(ValueError, match="dense"):
        ops.mxfp8_quantize(torch.zeros(64, 8, dtype=bf).t())
    with pytest.raises(ValueError, match="3-d"):
        ops.nvfp4_quantize_weight([x])
    with pytest.raises(ValueError, match="does not match"):
        ops.nvfp4_quantize_weight([torch.zeros(2, 64, 64, dtype=bf), torch.zeros(3, 64, 64, dtype=bf)])
    with pytest.raises(ValueError, match="CUDA"):
        ops.nvfp4_quantize_per_token(x)
    ids, prob = torch.zeros(4, 2, dtype=i32), torch.zeros(4, 2, dtype=f32)
    with pytest.raises(TypeError, match="topk_ids"):
        ops.moe_build_segments(ids.long(), prob, 8)
    with pytest.raises(ValueError, match="shape of topk_ids"):
        ops.moe_build_segments(ids, prob[:, :1], 8)
    with pytest.raises(ValueError, match="CUDA"):
        ops.moe_build_segments(ids, prob, 8)
    cap = ops.moe_row_capacity(4, 2, 8, 128)
    perm, seg = torch.zeros(cap, dtype=i32), torch.zeros(9, dtype=i32)
    with pytest.raises(ValueError, match="perm"):
        ops.moe_gather_bf16(x, perm[:10], seg, 8, 2, cap)
    with pytest.raises(ValueError, match="seg_offsets"):
        ops.moe_gather_bf16(x, perm, seg[:8], 8, 2, cap)
    with pytest.raises(ValueError, match="contiguous"):
        ops.moe_gather_bf16(torch.zeros(64, 8, dtype=bf).t(), perm, seg, 8, 2, cap)
    with pytest.raises(ValueError, match="CUDA"):
        ops.moe_gather_bf16(x, perm, seg, 8, 2, cap)
    q = torch.zeros(8, 32, dtype=u8)
    s = torch.zeros(ops.scale_bytes(8, 4), dtype=u8)
    ts = torch.zeros(8, dtype=f32)
    with pytest.raises(ValueError, match="codes"):
        ops.moe_gather_nvfp4(q, s, ts, 128, perm, seg, 8, 2, cap)
    with pytest.raises(ValueError, match="ts"):
        ops.moe_gather_nvfp4(q, s, ts[:4], 64, perm, seg, 8, 2, cap)
    with pytest.raises(ValueError, match="CUDA"):
        ops.moe_gather_nvfp4(q, s, ts, 64, perm, seg, 8, 2, cap)
    y, inv = torch.zeros(cap, 64, dtype=bf), torch.zeros(8, dtype=i32)
    with pytest.raises(ValueError, match="inv_perm"):
        ops.moe_combine(y, inv[:7], 4, 2)
    with pytest.raises(ValueError, match="out"):
        ops.moe_combine(y, inv, 4, 2, out=torch.zeros(3, 64, dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        ops.moe_combine(y, inv, 4, 2)


def test_binding_checks_gemm_and_dequantize_arguments(lib):
    """The GEMM wrapper checks element types the descriptor cannot carry:
    codes and scales uint8 (bf16 operands for the BF16 kind), fp32 output
    only for the fp32 epilogue, fp32 scales / probabilities / amax, int32
    offsets holding E+1 entries; the dequantisers check codes, scales and
    the device row count (CPU only)."""
    import torch
    from microscaled_precision_moe_gb300 import ops, _lib as L
    bf, i32, f32, u8 = torch.bfloat16, torch.int32, torch.float32, torch.uint8
    a, b = torch.zeros(256, 128, dtype=u8), torch.zeros(256, 128, dtype=u8)
    sf = torch.zeros(256 * 64, dtype=u8)
    seg = torch.zeros(3, dtype=i32)
    args = (L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, 2, 256, 256, 256)
    with pytest.raises(TypeError, match="a \\(codes\\)"):
        ops.moe_grouped_gemm(*args, seg, a.to(bf), b, sf, 16, sf, 16, torch.zeros(256, 256, dtype=bf))
    with pytest.raises(ValueError, match="scale tensors"):
        ops.moe_grouped_gemm(*args, seg, a, b, None, 16, sf, 16, torch.zeros(256, 256, dtype=bf))
    with pytest.raises(TypeError, match="out"):
        ops.moe_grouped_gemm(*args, seg, a, b, sf, 16, sf, 16, torch.zeros(256, 256, dtype=f32))
    with pytest.raises(TypeError, match="alpha_a"):
        ops.moe_grouped_gemm(*args, seg, a, b, sf, 16, sf, 16, torch.zeros(256, 256, dtype=bf),
                             alpha_a=torch.zeros(256, dtype=bf))
    with pytest.raises(ValueError, match="seg_offsets"):
        ops.moe_grouped_gemm(*args, seg[:2], a, b, sf, 16, sf, 16, torch.zeros(256, 256, dtype=bf))
    with pytest.raises(TypeError, match="out"):
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_K, L.EPI_F32, 2, 256, 256, 0, seg, a, b, sf, 16,
                             sf, 16, torch.zeros(2, 256, 256, dtype=bf))
    with pytest.raises(TypeError, match="b"):
        ops.moe_grouped_gemm(L.KIND_BF16, L.GROUP_M, L.EPI_BF16, 2, 256, 256, 256, seg,
                             torch.zeros(256, 256, dtype=bf), b, None, 0, None, 0,
                             torch.zeros(256, 256, dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        ops.moe_grouped_gemm(*args, seg, a, b, sf, 16, sf, 16, torch.zeros(256, 256, dtype=bf))
    q, s, ts = torch.zeros(8, 32, dtype=u8), torch.zeros(ops.scale_bytes(8, 4), dtype=u8), torch.zeros(8)
    with pytest.raises(TypeError, match="m_valid"):
        ops.nvfp4_dequantize(q, s, ts, 1, 64, m_valid=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(TypeError, match="out"):
        ops.nvfp4_dequantize(q, s, ts, 1, 64, out=torch.zeros(8, 64, dtype=f32))
    with pytest.raises(TypeError, match="amax_in"):
        ops.nvfp4_quantize_per_token(torch.zeros(8, 64, dtype=bf), amax_in=torch.zeros(8, dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        ops.mxfp8_dequantize(torch.zeros(8, 64, dtype=u8), torch.zeros(ops.scale_bytes(8, 2), dtype=u8))


def test_mxfp8_quantize_gather_validation(lib):
    """mpm_mxfp8_quantize_gather rejects bad arguments on the host."""
    fake = C.c_void_p(0x10000)
    odd = C.c_void_p(0x10008)
    f = lib.mpm_mxfp8_quantize_gather
    ok = dict(x=fake, T=4, K=64, ldx=64, perm=fake, k=2, seg=fake, E=2, cap=256, flags=3,
              rq=fake, rs=fake, cq=fake, ldc=256, cs=fake)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["T"], a["K"], a["ldx"], a["perm"], a["k"], a["seg"], a["E"], a["cap"],
                 a["flags"], a["rq"], a["rs"], a["cq"], a["ldc"], a["cs"], None)
    assert call(x=None) == 1 and call(perm=None) == 1 and call(seg=None) == 1
    assert call(rq=None) == 1 and call(cs=None) == 1
    assert call(flags=0) == 2 and call(flags=4) == 2
    assert call(T=0) == 2 and call(cap=0) == 2 and call(E=0) == 2
    assert call(k=0) == 2 and call(k=65) == 2
    assert call(K=16) == 2 and call(K=48) == 2 and call(ldx=32) == 2 and call(ldc=128) == 2
    assert call(ldx=1 << 31) == 2 and call(T=1 << 30, k=2) == 2
    assert call(x=odd) == 3 and call(ldx=68) == 3 and call(rq=odd) == 3
    assert call(cq=odd) == 3 and call(ldc=264) == 3
    # one copy only: the other copy's pointers are not needed
    assert call(flags=1, cq=None, cs=None, ldc=0, x=odd) == 3
    assert call(flags=2, rq=None, rs=None, x=odd) == 3


def test_quantize_scatter_validation(lib):
    """mpm_nvfp4_quantize_scatter rejects bad arguments on the host."""
    fake = C.c_void_p(0x10000)
    odd = C.c_void_p(0x10008)
    odd4 = C.c_void_p(0x10002)
    f = lib.mpm_nvfp4_quantize_scatter
    assert lib.mpm_nvfp4_quantize_scatter_workspace_bytes(4, 64) == 4 * 4 + 4 * 4 + 16
    assert lib.mpm_nvfp4_quantize_scatter_workspace_bytes(4, 96) == 0
    ok = dict(x=fake, T=4, K=64, ldx=64, inv=fake, k=2, perm=fake, seg=fake, E=2, cap=256,
              q=fake, s=fake, ts=fake, amax=None, ws=fake, wsb=48)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["T"], a["K"], a["ldx"], a["inv"], a["k"], a["perm"], a["seg"], a["E"],
                 a["cap"], a["q"], a["s"], a["ts"], a["amax"], a["ws"], a["wsb"], None)
    assert call(x=None) == 1 and call(inv=None) == 1 and call(ts=None) == 1 and call(ws=None) == 1
    assert call(wsb=47) == 2 and call(ws=odd4) == 3
    assert call(K=96) == 2 and call(K=16384, ldx=16384) == 2 and call(ldx=32) == 2
    assert call(k=0) == 2 and call(k=65) == 2 and call(T=0) == 2 and call(cap=0) == 2
    assert call(E=0) == 2
    assert call(x=odd) == 3 and call(q=odd) == 3 and call(ldx=68) == 3
    assert call(s=odd4) == 3 and call(amax=odd4) == 3
