"""Torch-facing wrappers of the libmpm C ABI (same names, minus the prefix).

PyTorch provides device memory and the current stream only; each function
allocates its outputs with torch and passes raw pointers to the library,
where every step runs in CUDA kernels.  Tensors must live on a CUDA device.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(dev=None):
    return C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmpm operates on CUDA tensors only")


def _check(t, name, dtype, dim=None, contiguous=False, min_numel=None):
    """Argument checks the C side cannot make (it sees raw pointers only):
    element type, rank, dense layout, and that a buffer holds at least the
    elements the call will touch."""
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name}: expected a {dim}-d tensor, got shape {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: holds {t.numel()} elements, the call needs {min_numel}")


def _check_m_valid(m_valid):
    """The optional device row count: one int32."""
    if m_valid is not None:
        _check(m_valid, "m_valid", torch.int32, min_numel=1)


def _check_rows(x, name):
    """A bf16 matrix whose rows are dense (any row pitch)."""
    _check(x, name, torch.bfloat16, dim=2)
    if x.stride(1) != 1:
        raise ValueError(f"{name}: rows must be dense (stride(1) == 1)")


def scale_bytes(rows: int, cols: int) -> int:
    return int(L.load().mpm_scale_bytes(rows, cols))


def pad_to(n: int, m: int) -> int:
    return (n + m - 1) // m * m


# ------------------------------------------------------------------ quantisers

def mxfp8_quantize(x, rowwise=True, colwise=True, ldc=None, m_valid=None, out=None):
    """MXFP8 row-wise 1x32 and/or column-wise 32x1 copies of bf16 x [M, K].

    Returns dict with row_q [M, K], row_s (tiled [M, K/32]), col_q [K, ldc]
    (transposed), col_s (tiled [K, ceil(M/32)]).
    """
    lib = L.load()
    _check_rows(x, "x")
    _check_m_valid(m_valid)
    _need_cuda(x, m_valid)
    M, K = x.shape
    ldc = ldc or pad_to(M, 16)
    dev = x.device
    o = out or {}
    flags = (L.ROWWISE if rowwise else 0) | (L.COLWISE if colwise else 0)
    if rowwise:
        o.setdefault("row_q", torch.empty(M, K, dtype=torch.uint8, device=dev))
        o.setdefault("row_s", torch.empty(scale_bytes(M, K // 32), dtype=torch.uint8, device=dev))
    if colwise:
        o.setdefault("col_q", torch.empty(K, ldc, dtype=torch.uint8, device=dev))
        o.setdefault("col_s", torch.empty(scale_bytes(K, (M + 31) // 32), dtype=torch.uint8,
                                          device=dev))
    st = lib.mpm_mxfp8_quantize(_ptr(x), M, K, x.stride(0), flags, _ptr(o.get("row_q")),
                                _ptr(o.get("row_s")), _ptr(o.get("col_q")), ldc,
                                _ptr(o.get("col_s")), _ptr(m_valid), _stream(dev))
    L.check(st, "mpm_mxfp8_quantize")
    return o


def mxfp8_quantize_gather(x, perm, seg, E: int, k: int, cap: int, rowwise=True, colwise=True,
                          ldc=None, out=None):
    """MXFP8 copies of the permuted layout of bf16 x [T, K] (cap rows, row r
    = token perm[r] // k, zero for padding rows), without the gathered bf16
    matrix: the bytes moe_gather_bf16 followed by mxfp8_quantize(...,
    m_valid=seg[E:]) give.  Same output dict as mxfp8_quantize with M = cap."""
    lib = L.load()
    _check_rows(x, "x")
    _check_route(perm, seg, E, cap)
    _need_cuda(x, perm, seg)
    T, K = x.shape
    ldc = ldc or pad_to(cap, 16)
    dev = x.device
    o = out or {}
    flags = (L.ROWWISE if rowwise else 0) | (L.COLWISE if colwise else 0)
    if rowwise:
        o.setdefault("row_q", torch.empty(cap, K, dtype=torch.uint8, device=dev))
        o.setdefault("row_s", torch.empty(scale_bytes(cap, K // 32), dtype=torch.uint8, device=dev))
    if colwise:
        o.setdefault("col_q", torch.empty(K, ldc, dtype=torch.uint8, device=dev))
        o.setdefault("col_s", torch.empty(scale_bytes(K, (cap + 31) // 32), dtype=torch.uint8,
                                          device=dev))
    st = lib.mpm_mxfp8_quantize_gather(_ptr(x), T, K, x.stride(0), _ptr(perm), k, _ptr(seg), E,
                                       cap, flags, _ptr(o.get("row_q")), _ptr(o.get("row_s")),
                                       _ptr(o.get("col_q")), ldc, _ptr(o.get("col_s")),
                                       _stream(dev))
    L.check(st, "mpm_mxfp8_quantize_gather")
    return o


def nvfp4_quantize_per_token(x, amax_in=None, m_valid=None, out=None):
    """Per-token NVFP4 of bf16 x [M, K]: (q [M, K/2] u8, s tiled [M, K/16] u8,
    token_scale [M] fp32) from one call."""
    lib = L.load()
    _check_rows(x, "x")
    _check_m_valid(m_valid)
    if amax_in is not None:
        _check(amax_in, "amax_in", torch.float32, min_numel=x.shape[0])
    _need_cuda(x, m_valid, amax_in)
    M, K = x.shape
    dev = x.device
    if out is None:
        out = (torch.empty(M, K // 2, dtype=torch.uint8, device=dev),
               torch.empty(scale_bytes(M, K // 16), dtype=torch.uint8, device=dev),
               torch.empty(M, dtype=torch.float32, device=dev))
    q, s, ts = out
    st = lib.mpm_nvfp4_quantize_per_token(_ptr(x), M, K, x.stride(0), _ptr(amax_in), _ptr(q),
                                          _ptr(s), _ptr(ts), _ptr(m_valid), _stream(dev))
    L.check(st, "mpm_nvfp4_quantize_per_token")
    return q, s, ts


def nvfp4_quantize_online(x, m_valid=None, out=None):
    """Tile-by-tile NVFP4 of bf16 x [M, K] with the running row amax (tiles
    of 256 columns): (q [M, K/2] u8, s tiled [M, K/16] u8, tile_scale
    [M, K/256] fp32)."""
    lib = L.load()
    _check_rows(x, "x")
    _check_m_valid(m_valid)
    _need_cuda(x, m_valid)
    M, K = x.shape
    if K % 256 != 0:
        raise ValueError(f"x: K = {K} is not a multiple of the 256-column tile")
    dev = x.device
    if out is None:
        out = (torch.empty(M, K // 2, dtype=torch.uint8, device=dev),
               torch.empty(scale_bytes(M, K // 16), dtype=torch.uint8, device=dev),
               torch.empty(M, K // 256, dtype=torch.float32, device=dev))
    q, s, gs = out
    _check(q, "q", torch.uint8, min_numel=M * (K // 2))
    _check(s, "s", torch.uint8, min_numel=scale_bytes(M, K // 16))
    _check(gs, "tile_scale", torch.float32, min_numel=M * (K // 256))
    st = lib.mpm_nvfp4_quantize_online(_ptr(x), M, K, x.stride(0), _ptr(q), _ptr(s), _ptr(gs),
                                       _ptr(m_valid), _stream(dev))
    L.check(st, "mpm_nvfp4_quantize_online")
    return q, s, gs


def nvfp4_quantize_weight(parts, out=None, ws=None):
    """Joint NVFP4 quantisation of per-expert parts [E, rows_p, K] (bf16) with
    one FP32 outer scale per expert: (q [E, R, K/2], s [E * tiled(R, K/16)],
    tensor_scale [E])."""
    lib = L.load()
    if not parts:
        raise ValueError("parts: at least one weight part is needed")
    for i, p in enumerate(parts):
        _check(p, f"parts[{i}]", torch.bfloat16, dim=3, contiguous=True)
    E, _, K = parts[0].shape
    for i, p in enumerate(parts):
        if p.shape[0] != E or p.shape[2] != K:
            raise ValueError(f"parts[{i}]: shape {tuple(p.shape)} does not match [{E}, rows, {K}]")
    _need_cuda(*parts)
    R = sum(p.shape[1] for p in parts)
    dev = parts[0].device
    if out is None:
        out = (torch.empty(E, R, K // 2, dtype=torch.uint8, device=dev),
               torch.empty(E * scale_bytes(R, K // 16), dtype=torch.uint8, device=dev),
               torch.empty(E, dtype=torch.float32, device=dev))
    q, s, ts = out
    wsb = int(lib.mpm_nvfp4_weight_workspace_bytes(E))
    if ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ptrs = (C.c_void_p * len(parts))(*[p.data_ptr() for p in parts])
    rows = (C.c_int64 * len(parts))(*[p.shape[1] for p in parts])
    st = lib.mpm_nvfp4_quantize_weight(ptrs, rows, len(parts), K, E, _ptr(q), _ptr(s), _ptr(ts),
                                       _ptr(ws), ws.numel(), _stream(dev))
    L.check(st, "mpm_nvfp4_quantize_weight")
    return q, s, ts


# ------------------------------------------------------------------ routing

def moe_row_capacity(T: int, k: int, E: int, pad: int = 128) -> int:
    return int(L.load().mpm_moe_row_capacity(T, k, E, pad))


def moe_build_segments(topk_ids, topk_prob, E: int, out=None, ws=None, pad: int = 128):
    """(seg_offsets [E+1], perm [cap], inv_perm [T*k], row_prob [cap], cap);
    segments padded to ``pad`` rows (128, or 256 for the CTA-pair GEMM)."""
    lib = L.load()
    _check(topk_ids, "topk_ids", torch.int32, dim=2)
    _check(topk_prob, "topk_prob", torch.float32, dim=2)
    if topk_prob.shape != topk_ids.shape:
        raise ValueError("topk_prob must have the shape of topk_ids")
    _need_cuda(topk_ids, topk_prob)
    ids_c, prob_c = topk_ids.contiguous(), topk_prob.contiguous()   # alive until the launch
    T, k = topk_ids.shape
    dev = topk_ids.device
    cap = moe_row_capacity(T, k, E, pad)
    if out is None:
        out = (torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(cap, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(cap, dtype=torch.float32, device=dev))
    seg, perm, inv, rp = out
    wsb = int(lib.mpm_moe_segments_workspace_bytes(T, k, E))
    if ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    _check(seg, "seg_offsets", torch.int32, min_numel=E + 1)
    _check(perm, "perm", torch.int32, min_numel=cap)
    _check(inv, "inv_perm", torch.int32, min_numel=T * k)
    _check(rp, "row_prob", torch.float32, min_numel=cap)
    _check(ws, "ws", torch.uint8, min_numel=wsb)
    st = lib.mpm_moe_build_segments(_ptr(ids_c), _ptr(prob_c), T,
                                    k, E, pad, _ptr(seg), _ptr(perm), _ptr(inv), _ptr(rp),
                                    _ptr(ws), ws.numel(), _stream(dev))
    L.check(st, "mpm_moe_build_segments")
    return seg, perm, inv, rp, cap


def _check_route(perm, seg, E, cap):
    _check(perm, "perm", torch.int32, min_numel=cap)
    _check(seg, "seg_offsets", torch.int32, min_numel=E + 1)


def moe_gather_bf16(x, perm, seg, E: int, k: int, cap: int, out=None, amax_zero=None):
    """bf16 rows x [T, K] (dense) -> the permuted layout [cap, K]."""
    lib = L.load()
    _check(x, "x", torch.bfloat16, dim=2, contiguous=True)
    _check_route(perm, seg, E, cap)
    T, K = x.shape
    if out is None:
        out = torch.empty(cap, K, dtype=torch.bfloat16, device=x.device)
    _check(out, "out", torch.bfloat16, contiguous=True, min_numel=cap * K)
    if amax_zero is not None:
        _check(amax_zero, "amax_zero", torch.float32, min_numel=cap)
    _need_cuda(x, perm, seg, out, amax_zero)
    st = lib.mpm_moe_gather(L.GATHER_BF16, _ptr(x), None, None, T, K, k, _ptr(perm), _ptr(seg),
                            E, cap, _ptr(out), None, None, _ptr(amax_zero), _stream(x.device))
    L.check(st, "mpm_moe_gather")
    return out


def nvfp4_quantize_scatter_workspace_bytes(T: int, K: int) -> int:
    return int(L.load().mpm_nvfp4_quantize_scatter_workspace_bytes(T, K))


def nvfp4_quantize_scatter(x, inv_perm, perm, seg, E: int, k: int, cap: int, out=None,
                           amax_zero=None, ws=None):
    """Per-token NVFP4 of bf16 x [T, K] written straight into the permuted
    layout of cap rows: (codes [cap, K/2], tiled scales, token scales [cap]),
    the bytes nvfp4_quantize_per_token followed by moe_gather_nvfp4 give.
    ws: uint8 workspace of nvfp4_quantize_scatter_workspace_bytes(T, K)."""
    lib = L.load()
    _check_rows(x, "x")
    T, K = x.shape
    need = nvfp4_quantize_scatter_workspace_bytes(T, K)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(ws, "ws", torch.uint8, min_numel=need)
    _check(inv_perm, "inv_perm", torch.int32, min_numel=T * k)
    _check_route(perm, seg, E, cap)
    dev = x.device
    if out is None:
        out = (torch.empty(cap, K // 2, dtype=torch.uint8, device=dev),
               torch.empty(scale_bytes(cap, K // 16), dtype=torch.uint8, device=dev),
               torch.empty(cap, dtype=torch.float32, device=dev))
    dq, ds, dts = out
    _check(dq, "out codes", torch.uint8, contiguous=True, min_numel=cap * (K // 2))
    _check(ds, "out scales", torch.uint8, min_numel=scale_bytes(cap, K // 16))
    _check(dts, "out token scales", torch.float32, min_numel=cap)
    if amax_zero is not None:
        _check(amax_zero, "amax_zero", torch.float32, min_numel=cap)
    _need_cuda(x, inv_perm, perm, seg, dq, ds, dts, amax_zero, ws)
    st = lib.mpm_nvfp4_quantize_scatter(_ptr(x), T, K, x.stride(0), _ptr(inv_perm), k,
                                        _ptr(perm), _ptr(seg), E, cap, _ptr(dq), _ptr(ds),
                                        _ptr(dts), _ptr(amax_zero), _ptr(ws), ws.numel(),
                                        _stream(dev))
    L.check(st, "mpm_nvfp4_quantize_scatter")
    return dq, ds, dts


def moe_gather_nvfp4(q, s, ts, K: int, perm, seg, E: int, k: int, cap: int, out=None,
                     amax_zero=None):
    """Per-token NVFP4 rows (codes [T, K/2], tiled scales, token scales [T])
    -> the same three in the permuted layout of cap rows."""
    lib = L.load()
    _check(q, "q", torch.uint8, dim=2, contiguous=True)
    T = q.shape[0]
    if q.shape[1] != K // 2:
        raise ValueError(f"q: expected [T, {K // 2}] codes, got {tuple(q.shape)}")
    _check(s, "s", torch.uint8, min_numel=scale_bytes(T, K // 16))
    _check(ts, "ts", torch.float32, min_numel=T)
    _check_route(perm, seg, E, cap)
    dev = q.device
    if out is None:
        out = (torch.empty(cap, K // 2, dtype=torch.uint8, device=dev),
               torch.empty(scale_bytes(cap, K // 16), dtype=torch.uint8, device=dev),
               torch.empty(cap, dtype=torch.float32, device=dev))
    dq, ds, dts = out
    _check(dq, "out codes", torch.uint8, contiguous=True, min_numel=cap * (K // 2))
    _check(ds, "out scales", torch.uint8, min_numel=scale_bytes(cap, K // 16))
    _check(dts, "out token scales", torch.float32, min_numel=cap)
    if amax_zero is not None:
        _check(amax_zero, "amax_zero", torch.float32, min_numel=cap)
    _need_cuda(q, s, ts, perm, seg, dq, ds, dts, amax_zero)
    st = lib.mpm_moe_gather(L.GATHER_NVFP4, _ptr(q), _ptr(s), _ptr(ts), T, K, k, _ptr(perm),
                            _ptr(seg), E, cap, _ptr(dq), _ptr(ds), _ptr(dts), _ptr(amax_zero),
                            _stream(dev))
    L.check(st, "mpm_moe_gather")
    return dq, ds, dts


def moe_combine(y_perm, inv_perm, T: int, k: int, out=None):
    """out [T, H] bf16: each token's k rows of y_perm summed in slot order."""
    lib = L.load()
    _check(y_perm, "y_perm", torch.bfloat16, dim=2, contiguous=True)
    _check(inv_perm, "inv_perm", torch.int32, min_numel=T * k)
    H = y_perm.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=y_perm.device)
    _check(out, "out", torch.bfloat16, contiguous=True, min_numel=T * H)
    _need_cuda(y_perm, inv_perm, out)
    st = lib.mpm_moe_combine(_ptr(y_perm), _ptr(inv_perm), T, k, H, _ptr(out),
                             _stream(y_perm.device))
    L.check(st, "mpm_moe_combine")
    return out


# ------------------------------------------------------------------ GEMM

def moe_grouped_gemm(kind, group, epilogue, E, a_rows, N, K, seg, a, b, sfa, sfa_cols, sfb,
                     sfb_cols, out, b_rows_per_expert=0, b_k_per_expert=0, alpha_a=None,
                     alpha_b=None, row_prob=None, out2=None, aux=None, amax=None, tile_m=128,
                     a_mn_major=False, b_mn_major=False, row_perm=None):
    """One grouped block-scaled GEMM launch (see mpm_grouped_gemm_desc).

    a, b: uint8 code matrices [rows, pitch bytes] (bf16 matrices [rows, K]
    for KIND_BF16, sfa / sfb None; with a_mn_major / b_mn_major the bf16
    matrix is [K rows, M or N]); out / out2 / aux: row-major
    tensors whose row strides become ldo / ldo2 / ld_aux.  row_perm: the
    segment build's row map; padding rows' outputs may then be left
    unwritten (small-M kernel).
    """
    lib = L.load()
    if kind == L.KIND_BF16:
        _check(a, "a", torch.bfloat16, dim=2)
        _check(b, "b", torch.bfloat16)
    else:
        _check(a, "a (codes)", torch.uint8, dim=2)
        _check(b, "b (codes)", torch.uint8)
        if sfa is None or sfb is None:
            raise ValueError("block-scaled kinds need both scale tensors")
        _check(sfa, "sfa", torch.uint8)
        _check(sfb, "sfb", torch.uint8)
    _check(out, "out", torch.float32 if epilogue == L.EPI_F32 else torch.bfloat16)
    if out2 is not None:
        _check(out2, "out2", torch.bfloat16)
    if aux is not None:
        if epilogue == L.EPI_BF16_ONLINE:
            # the per-(row, 256-column tile) outer scales of the online quantiser
            _check(aux, "aux (tile scales)", torch.float32, dim=2)
            if aux.shape[0] < a_rows or aux.shape[1] < K // 256:
                raise ValueError(f"aux: shape {tuple(aux.shape)}, the call needs "
                                 f"[{a_rows}, {K // 256}]")
        else:
            _check(aux, "aux", torch.bfloat16)
    for t, name in ((alpha_a, "alpha_a"), (alpha_b, "alpha_b"), (row_prob, "row_prob"),
                    (amax, "amax")):
        if t is not None:
            _check(t, name, torch.float32)
    if seg is not None:
        _check(seg, "seg_offsets", torch.int32, min_numel=E + 1)
    if row_perm is not None:
        _check(row_perm, "row_perm", torch.int32, min_numel=a_rows)
    _need_cuda(a, b, sfa, sfb, out, out2, aux, alpha_a, alpha_b, row_prob, amax, seg, row_perm)
    d = L.GroupedGemmDesc()
    d.kind, d.group, d.epilogue, d.tile_m = kind, group, epilogue, tile_m
    d.E, d.a_rows, d.N, d.K = E, a_rows, N, K
    d.seg_dev = None if seg is None else seg.data_ptr()
    d.a_dev, d.a_total_rows = a.data_ptr(), a.shape[0]
    d.lda_bytes = a.stride(0) * a.element_size()
    d.b_dev, d.ldb_bytes = b.data_ptr(), b.stride(-2) * b.element_size()
    d.b_total_rows = b.numel() // b.stride(-2)
    d.b_rows_per_expert, d.b_k_per_expert = b_rows_per_expert, b_k_per_expert
    d.sfa_dev, d.sfa_cols = (None if sfa is None else sfa.data_ptr()), sfa_cols
    d.sfb_dev, d.sfb_cols = (None if sfb is None else sfb.data_ptr()), sfb_cols
    d.alpha_a_dev = None if alpha_a is None else alpha_a.data_ptr()
    d.alpha_b_dev = None if alpha_b is None else alpha_b.data_ptr()
    d.row_prob_dev = None if row_prob is None else row_prob.data_ptr()
    d.out_dev, d.ldo = out.data_ptr(), out.stride(-2)
    if out2 is not None:
        d.out2_dev, d.ldo2 = out2.data_ptr(), out2.stride(-2)
    if aux is not None:
        d.aux_dev, d.ld_aux = aux.data_ptr(), aux.stride(-2)
    d.amax_dev = None if amax is None else amax.data_ptr()
    d.a_mn_major, d.b_mn_major = int(bool(a_mn_major)), int(bool(b_mn_major))
    d.row_perm_dev = None if row_perm is None else row_perm.data_ptr()
    if group == L.GROUP_K:
        # the weight-gradient form has its own entry point
        st = lib.mpm_moe_grouped_gemm_wgrad(C.byref(d), _stream(a.device))
        L.check(st, "mpm_moe_grouped_gemm_wgrad")
    else:
        st = lib.mpm_moe_grouped_gemm(C.byref(d), _stream(a.device))
        L.check(st, "mpm_moe_grouped_gemm")
    return out


# ------------------------------------------------------------ BF16 backward operands

def nvfp4_dequantize(q, s, outer, rows_per_outer: int, K: int, m_valid=None, out=None):
    """bf16 [M, K] from NVFP4 codes, tiled E4M3 scales and fp32 outer scales
    (one outer scale per ``rows_per_outer`` rows), each value rounded once."""
    lib = L.load()
    _check(q, "q", torch.uint8, dim=2)
    _check(s, "s", torch.uint8)
    _check(outer, "outer", torch.float32)
    _check_m_valid(m_valid)
    M = q.shape[0]
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, dim=2)
    _need_cuda(q, s, outer, m_valid, out)
    st = lib.mpm_nvfp4_dequantize(_ptr(q), _ptr(s), _ptr(outer), rows_per_outer, M, K,
                                  _ptr(out), out.stride(0), _ptr(m_valid), _stream(q.device))
    L.check(st, "mpm_nvfp4_dequantize")
    return out


def mxfp8_dequantize(q, s, m_valid=None, out=None):
    """bf16 [M, K] from row-wise MXFP8 codes [M, K] and tiled E8M0 scales."""
    lib = L.load()
    _check(q, "q", torch.uint8, dim=2)
    _check(s, "s", torch.uint8)
    _check_m_valid(m_valid)
    M, K = q.shape
    if out is None:
        out = torch.empty(M, K, dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, dim=2)
    _need_cuda(q, s, m_valid, out)
    st = lib.mpm_mxfp8_dequantize(_ptr(q), _ptr(s), M, K, _ptr(out), out.stride(0),
                                  _ptr(m_valid), _stream(q.device))
    L.check(st, "mpm_mxfp8_dequantize")
    return out


def transpose_bf16(x, m_valid=None, out=None):
    """out [C, R] = x [R, C]^T for bf16 matrices (bit copies)."""
    lib = L.load()
    _check(x, "x", torch.bfloat16, dim=2)
    _check_m_valid(m_valid)
    R, C_ = x.shape
    if out is None:
        out = torch.empty(C_, R, dtype=torch.bfloat16, device=x.device)
    _check(out, "out", torch.bfloat16, dim=2)
    _need_cuda(x, m_valid, out)
    st = lib.mpm_transpose_bf16(_ptr(x), R, C_, x.stride(0), _ptr(out), out.stride(0),
                                _ptr(m_valid), _stream(x.device))
    L.check(st, "mpm_transpose_bf16")
    return out


def get_device_status() -> int:
    lib = L.load()
    v = C.c_int32(0)
    L.check(lib.mpm_get_device_status(C.byref(v), _stream()), "mpm_get_device_status")
    return int(v.value)
