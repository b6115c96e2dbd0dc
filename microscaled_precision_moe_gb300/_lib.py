"""ctypes binding of libmpm (the C ABI declared in include/mpm.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Loading fails loudly when the library has not been built; there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmpm.so")

MPM_OK = 0
STATUS_NAMES = {0: "MPM_OK", 1: "MPM_ERR_NULL", 2: "MPM_ERR_SHAPE", 3: "MPM_ERR_ALIGN",
                4: "MPM_ERR_UNSUPPORTED", 5: "MPM_ERR_CUDA", 6: "MPM_ERR_DEVICE_TIMEOUT",
                7: "MPM_ERR_DEVICE_BOUNDS"}

ROWWISE, COLWISE = 1, 2
KIND_NVFP4, KIND_MXFP8, KIND_BF16 = 0, 1, 2
GROUP_M, GROUP_K = 0, 1
TILE_SMALL_M = 1
EPI_F32, EPI_BF16, EPI_SWIGLU, EPI_SWIGLU_SAVE, EPI_DSWIGLU, EPI_BF16_ONLINE = 0, 1, 2, 3, 4, 5
GATHER_BF16, GATHER_NVFP4 = 0, 1

_vp, _i64, _u32, _int, _sz = C.c_void_p, C.c_int64, C.c_uint, C.c_int, C.c_size_t


class GroupedGemmDesc(C.Structure):
    """Mirror of mpm_grouped_gemm_desc."""
    _fields_ = [
        ("kind", _int), ("tile_m", _int), ("group", _int), ("epilogue", _int),
        ("E", _i64), ("a_rows", _i64), ("N", _i64), ("K", _i64),
        ("seg_dev", _vp),
        ("a_dev", _vp), ("lda_bytes", _i64), ("a_total_rows", _i64),
        ("b_dev", _vp), ("ldb_bytes", _i64), ("b_total_rows", _i64),
        ("b_rows_per_expert", _i64), ("b_k_per_expert", _i64),
        ("sfa_dev", _vp), ("sfa_cols", _i64),
        ("sfb_dev", _vp), ("sfb_cols", _i64),
        ("alpha_a_dev", _vp), ("alpha_b_dev", _vp), ("row_prob_dev", _vp),
        ("out_dev", _vp), ("ldo", _i64),
        ("out2_dev", _vp), ("ldo2", _i64),
        ("aux_dev", _vp), ("ld_aux", _i64),
        ("amax_dev", _vp),
        ("a_mn_major", _int), ("b_mn_major", _int),
        ("row_perm_dev", _vp),
    ]


_SIGS = {
    "mpm_status_string": (C.c_char_p, [_int]),
    "mpm_version": (_int, []),
    "mpm_scale_bytes": (_sz, [_i64, _i64]),
    "mpm_mxfp8_quantize": (_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp, _i64, _vp, _vp, _vp]),
    "mpm_mxfp8_quantize_gather": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _vp, _i64, _i64, _u32,
                                         _vp, _vp, _vp, _i64, _vp, _vp]),
    "mpm_nvfp4_quantize_per_token": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mpm_nvfp4_quantize_online": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "mpm_nvfp4_weight_workspace_bytes": (_sz, [_i64]),
    "mpm_nvfp4_quantize_weight": (_int, [C.POINTER(_vp), C.POINTER(_i64), _int, _i64, _i64,
                                         _vp, _vp, _vp, _vp, _sz, _vp]),
    "mpm_nvfp4_quantize_weight_noalloc": (_int, [C.POINTER(_vp), C.POINTER(_i64), _int, _i64,
                                                 _i64, _vp, _vp, _vp, _vp]),
    "mpm_moe_row_capacity": (_i64, [_i64, _int, _i64, _int]),
    "mpm_moe_segments_workspace_bytes": (_sz, [_i64, _int, _i64]),
    "mpm_moe_build_segments": (_int, [_vp, _vp, _i64, _int, _i64, _int, _vp, _vp, _vp, _vp, _vp,
                                      _sz, _vp]),
    "mpm_moe_gather": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _int, _vp, _vp, _i64, _i64,
                              _vp, _vp, _vp, _vp, _vp]),
    "mpm_moe_combine": (_int, [_vp, _vp, _i64, _int, _i64, _vp, _vp]),
    "mpm_nvfp4_quantize_scatter_workspace_bytes": (C.c_size_t, [_i64, _i64]),
    "mpm_nvfp4_quantize_scatter": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _vp, _vp, _i64,
                                          _i64, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp]),
    "mpm_nvfp4_dequantize": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]),
    "mpm_mxfp8_dequantize": (_int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "mpm_transpose_bf16": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]),
    "mpm_moe_grouped_gemm": (_int, [C.POINTER(GroupedGemmDesc), _vp]),
    "mpm_moe_grouped_gemm_wgrad": (_int, [C.POINTER(GroupedGemmDesc), _vp]),
    "mpm_get_device_status": (_int, [C.POINTER(C.c_int32), _vp]),
}

EXPORTED = tuple(_SIGS)

_lib = None


class MpmError(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Load libmpm.so (build it first with ``python -m
    microscaled_precision_moe_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise MpmError(f"libmpm.so not found at {path}; build it with "
                       f"`python -m microscaled_precision_moe_gb300.build`")
    lib = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str = ""):
    if status != MPM_OK:
        raise MpmError(f"{what}: {STATUS_NAMES.get(status, status)}")
