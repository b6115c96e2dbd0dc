"""MoE expert layer on the libmpm kernels: NVFP4 forward, MXFP8 forward+backward.

Every step of both paths runs in the library's CUDA kernels; this module only
owns the buffers (allocated once per shape, reused every step) and sequences
the calls on the current stream.  No host synchronisation happens inside a
step: expert offsets stay on the device.

NVFP4 forward ("miniTE technical report", sections 5.2-5.4; "Towards
Blackwell-native 8-bit and 4-bit RL", section "Per-token activation
scaling"):
  X --per-token NVFP4, written straight into the expert-ordered rows--> A
     (codes, block scales, token scale; the same bytes as quantising then
     gathering by expert)
  A x W1[e]^T  (gate|up)  --epilogue: alpha, SwiGLU x prob, row amax--> D (bf16)
  D --per-token NVFP4 reusing the amax--> A2
  A2 x W2[e]^T --epilogue: alpha--> Y_perm (bf16) --combine--> out (bf16)

BF16 backward of the NVFP4 layer ("Towards Blackwell-native 8-bit and 4-bit
RL", section "High-precision and dequantized backward"): the four backward
GEMMs run on the tensor cores in BF16 (fp32 accumulation), either on the
original BF16 operands ("high_precision") or on the BF16 dequantisation of
exactly the NVFP4 operands the forward consumed ("dequantized"):
  dY --gather--> dY_perm;  dY_perm x W2^T-copy --epilogue: SwiGLU backward--> dH
  dY_perm^T x D per expert --> dW2;  dH x W1^T-copy --> dX_perm --combine--> dX
  dH^T x X_perm per expert --> dW1

MXFP8 forward + backward ("Towards Blackwell-native 8-bit and 4-bit RL",
section "Recipe 1 / Training"): every GEMM operand is quantised from bf16;
fprop uses row-wise copies, dgrad the row-wise gradient and the column-wise
weight copy, wgrad the column-wise gradient and activation copies.  X and dY
are quantised straight from their token rows into the expert-ordered row-wise
and column-wise copies (the same bytes as gathering by expert, then
quantising), so no permuted bf16 copy is written.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib as L
from . import ops


def _sb(rows, cols):
    return ops.scale_bytes(rows, cols)


def _bf16_backward_gemms(L_, x_op, d_op, w1_op, w2_op, dy, mark, m0):
    """The BF16 backward of an expert layer on given operands (both layers):
    gather dY, FC2 dgrad with the SwiGLU backward fused, FC2 wgrad, FC1
    dgrad, combine, FC1 wgrad — every operand read row-major (MN-major where
    the GEMM contracts over rows).  Buffers (dyp, dh, dxp, dx, dw1, dw2, c1,
    seg) belong to the layer ``L_``; ``mark(m0 + i)`` before each stage."""
    T, H, I, E, k, cap = L_.T, L_.H, L_.I, L_.E, L_.k, L_.cap
    seg, perm, inv, rp = L_.seg
    bf = L.KIND_BF16
    mark(m0)
    ops.moe_gather_bf16(dy, perm, seg, E, k, cap, out=L_.dyp)
    mark(m0 + 1)
    ops.moe_grouped_gemm(bf, L.GROUP_M, L.EPI_DSWIGLU, E, cap, I, H, seg, L_.dyp, w2_op,
                         None, 0, None, 0, L_.dh, b_rows_per_expert=0, b_k_per_expert=H,
                         row_prob=rp, aux=L_.c1, tile_m=256, b_mn_major=True)
    mark(m0 + 2)
    ops.moe_grouped_gemm(bf, L.GROUP_K, L.EPI_F32, E, H, I, 0, seg, L_.dyp, d_op,
                         None, 0, None, 0, L_.dw2, tile_m=256, a_mn_major=True, b_mn_major=True)
    mark(m0 + 3)
    ops.moe_grouped_gemm(bf, L.GROUP_M, L.EPI_BF16, E, cap, H, 2 * I, seg, L_.dh, w1_op,
                         None, 0, None, 0, L_.dxp, b_rows_per_expert=0, b_k_per_expert=2 * I,
                         tile_m=256, b_mn_major=True)
    mark(m0 + 4)
    ops.moe_combine(L_.dxp, inv, T, k, out=L_.dx)
    mark(m0 + 5)
    ops.moe_grouped_gemm(bf, L.GROUP_K, L.EPI_F32, E, 2 * I, H, 0, seg, L_.dh, x_op,
                         None, 0, None, 0, L_.dw1, tile_m=256, a_mn_major=True, b_mn_major=True)
    mark(m0 + 6)
    return L_.dx, L_.dw1, L_.dw2


# ============================================================================
# NVFP4
# ============================================================================

@dataclass
class NVFP4Weights:
    """Quantised expert weights: W1 = gate|up [E, 2I, H/2] with one outer scale
    per expert shared by gate and up, W2 [E, H, I/2]."""
    w1_q: torch.Tensor
    w1_s: torch.Tensor
    w1_ts: torch.Tensor
    w2_q: torch.Tensor
    w2_s: torch.Tensor
    w2_ts: torch.Tensor
    E: int
    H: int
    I: int

    @staticmethod
    def quantize(w1: torch.Tensor, w2: torch.Tensor) -> "NVFP4Weights":
        E, I2, H = w1.shape
        I = I2 // 2
        # W1 [E, 2I, H] already holds each expert's gate rows then up rows, so
        # one part of 2I rows per expert gives the joint gate/up scale
        q1, s1, t1 = ops.nvfp4_quantize_weight([w1.contiguous()])
        q2, s2, t2 = ops.nvfp4_quantize_weight([w2.contiguous()])
        return NVFP4Weights(q1, s1, t1, q2, s2, t2, E, H, I)


class NVFP4MoE:
    """Buffers and launch sequence of the NVFP4 expert-layer forward for a
    fixed (T, H, I, E, k).  tile_m = 256 (default) runs the grouped GEMMs on
    CTA pairs and pads expert segments to 256 rows; 128 uses one CTA per
    128-row tile and 128-row segments; L.TILE_SMALL_M (1) runs the small-M
    kernel (weights on the MMA's M side) for decode / rollout batches where
    each expert receives few rows, with 128-row segments.

    fc2 = "online" (CTA pairs only) runs FC2 as in the single-pass FFN of the
    miniTE report, section 5.6: D is quantised tile by tile (256 columns)
    against a running row amax, and FC2 weighs each tile's product by that
    tile's outer scale; fc2 = "two_pass" (default) re-quantises whole rows of
    D against their full amax."""

    FC2_MODES = ("two_pass", "online")

    def __init__(self, T, H, I, E, k, device="cuda", tile_m=256, fc2="two_pass"):
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        if fc2 not in self.FC2_MODES:
            raise ValueError(f"fc2 must be one of {self.FC2_MODES}")
        if fc2 == "online" and (tile_m != 256 or I % 256 != 0):
            raise ValueError("the online FC2 needs tile_m = 256 and I % 256 == 0")
        self.fc2 = fc2
        self.tile_m = tile_m
        self.pad = 128 if tile_m == L.TILE_SMALL_M else tile_m
        dev = torch.device(device)
        cap = ops.moe_row_capacity(T, k, E, self.pad)
        self.cap = cap
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda *s, dtype: torch.empty(*s, dtype=dtype, device=dev)
        self.seg = (e(E + 1, dtype=torch.int32), e(cap, dtype=torch.int32),
                    e(T * k, dtype=torch.int32), e(cap, dtype=f32))
        self.seg_ws = e(int(L.load().mpm_moe_segments_workspace_bytes(T, k, E)), dtype=u8)
        self.aq = (e(cap, H // 2, dtype=u8), e(_sb(cap, H // 16), dtype=u8), e(cap, dtype=f32))
        self.xq_ws = e(ops.nvfp4_quantize_scatter_workspace_bytes(T, H), dtype=u8)
        self.d = e(cap, I, dtype=bf)
        self.amax = e(cap, dtype=f32)
        # two-pass: one outer scale per row; online: one per (row, 256-column tile)
        self.dq = (e(cap, I // 2, dtype=u8), e(_sb(cap, I // 16), dtype=u8),
                   e(cap, dtype=f32) if fc2 == "two_pass" else e(cap, I // 256, dtype=f32))
        self.y = e(cap, H, dtype=bf)
        self.out = e(T, H, dtype=bf)

    # each call below is one or more library launches on the current stream
    # (quant_x: each token quantised once, straight into its k routed rows)
    STAGES = ("segments", "quant_x", "fc1", "quant_d", "fc2", "combine")

    def forward(self, x, topk_ids, topk_prob, w: NVFP4Weights, mark=None,
                save_for_backward=False, out=None, out_chunks=1, on_chunk=None):
        """out [T, H] bf16 (the layer's own buffer, or ``out`` when given).
        ``mark(i)`` (optional) is called before stage i of STAGES and once
        more at the end (used to record CUDA events).  save_for_backward: the
        FC1 epilogue also stores C = gate|up (bf16, [capacity, 2I]) for the
        SwiGLU backward.  out_chunks > 1 combines the output in that many
        contiguous token ranges, and ``on_chunk(j, t0, t1)`` (optional) is
        called right after range j = [t0, t1) is launched on the current
        stream, so a caller can record an event there and start copying
        those rows out while the later ranges are combined.  The result is
        the same bytes: each token's combine is independent of the others.
        self.y holds FC2's output for the routed rows; with the small-M
        kernel a segment's padding rows of it are left unwritten."""
        T, H, I, E, k, cap = self.T, self.H, self.I, self.E, self.k, self.cap
        mark = mark or (lambda i: None)
        mark(0)
        seg, perm, inv, rp = self.seg
        ops.moe_build_segments(topk_ids, topk_prob, E, out=self.seg, ws=self.seg_ws,
                               pad=self.pad)
        mark(1)
        ops.nvfp4_quantize_scatter(x, inv, perm, seg, E, k, cap, out=self.aq, amax_zero=self.amax,
                                   ws=self.xq_ws)
        aq, as_, ats = self.aq
        mark(2)
        if save_for_backward:
            self._alloc_backward()
        epi, c_out = (L.EPI_SWIGLU_SAVE, self.c1) if save_for_backward else (L.EPI_SWIGLU, self.d)
        ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, epi, E, cap, 2 * I, H, seg,
                             aq, w.w1_q.view(E * 2 * I, H // 2), as_, H // 16, w.w1_s, H // 16,
                             c_out, b_rows_per_expert=2 * I, alpha_a=ats, alpha_b=w.w1_ts,
                             row_prob=rp, out2=self.d, amax=self.amax, tile_m=self.tile_m)
        mark(3)
        if self.fc2 == "online":
            ops.nvfp4_quantize_online(self.d, m_valid=seg[E:], out=self.dq)
        else:
            ops.nvfp4_quantize_per_token(self.d, amax_in=self.amax, m_valid=seg[E:], out=self.dq)
        dq, ds, dts = self.dq
        mark(4)
        if self.fc2 == "online":
            ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16_ONLINE, E, cap, H, I, seg,
                                 dq, w.w2_q.view(E * H, I // 2), ds, I // 16, w.w2_s, I // 16,
                                 self.y, b_rows_per_expert=H, alpha_b=w.w2_ts, aux=dts,
                                 tile_m=256)
        else:
            ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                                 dq, w.w2_q.view(E * H, I // 2), ds, I // 16, w.w2_s, I // 16,
                                 self.y, b_rows_per_expert=H, alpha_a=dts, alpha_b=w.w2_ts,
                                 row_perm=perm,
                                 tile_m=self.tile_m)
        mark(5)
        dst = self.out if out is None else out
        n = max(1, min(int(out_chunks), T))
        for j in range(n):
            t0, t1 = j * T // n, (j + 1) * T // n
            ops.moe_combine(self.y, inv[t0 * k:t1 * k], t1 - t0, k, out=dst[t0:t1])
            if on_chunk is not None:
                on_chunk(j, t0, t1)
        mark(6)
        return dst

    # kernels launched by one forward: the segment build (one cooperative
    # kernel, after an 8-byte memset of its barrier words), the quantiser into
    # the routed rows (two kernels), FC1, the quantiser of D, FC2, combine
    LAUNCHES_PER_FORWARD = 7

    # ------------------------------------------------------------ BF16 backward
    BACKWARD_MODES = ("high_precision", "dequantized")
    BACKWARD_STAGES = ("operands", "gather_dy", "fc2_dgrad", "fc2_wgrad", "fc1_dgrad",
                       "combine", "fc1_wgrad")

    def _alloc_backward(self):
        if getattr(self, "c1", None) is not None:
            return
        T, H, I, E, cap = self.T, self.H, self.I, self.E, self.cap
        dev = self.d.device
        bf, f32 = torch.bfloat16, torch.float32
        e = lambda *s, dtype=bf: torch.empty(*s, dtype=dtype, device=dev)
        self.c1 = e(cap, 2 * I)
        self.xp = e(cap, H)              # X operand of the FC1 wgrad (per mode)
        self.dop = e(cap, I)             # dequantised D (dequantized mode)
        self.dyp = e(cap, H)
        self.dh = e(cap, 2 * I)
        self.dxp = e(cap, H)
        self.dx = e(T, H)
        self.dw1 = e(E, 2 * I, H, dtype=f32)
        self.dw2 = e(E, H, I, dtype=f32)
        self.w1_op = None                # [E*2I, H] bf16 weight operands of the dgrads
        self.w2_op = None                # [E*H, I]
        self._wq_op = None

    def prepare_backward_weights(self, mode, w1=None, w2=None, w: NVFP4Weights = None):
        """Weight operands of the dgrad GEMMs, once per weight update: the BF16
        weights themselves (high_precision, w1 / w2 given), or the BF16
        dequantisation of the NVFP4 weights the forward used (dequantized, w
        given).  The GEMMs read them row-major (MN-major B), no transposes."""
        self._alloc_backward()
        E, H, I = self.E, self.H, self.I
        if mode == "high_precision":
            self.w1_op, self.w2_op = w1.reshape(E * 2 * I, H), w2.reshape(E * H, I)
        elif mode == "dequantized":
            if self._wq_op is None:
                dev = self.d.device
                self._wq_op = (torch.empty(E * 2 * I, H, dtype=torch.bfloat16, device=dev),
                               torch.empty(E * H, I, dtype=torch.bfloat16, device=dev))
            self.w1_op = ops.nvfp4_dequantize(w.w1_q.view(E * 2 * I, H // 2), w.w1_s, w.w1_ts,
                                              2 * I, H, out=self._wq_op[0])
            self.w2_op = ops.nvfp4_dequantize(w.w2_q.view(E * H, I // 2), w.w2_s, w.w2_ts, H, I,
                                              out=self._wq_op[1])
        else:
            raise ValueError(f"unknown backward mode {mode!r}")
        self._w_mode = mode

    def backward(self, dy, mode, x=None, mark=None):
        """dX [T, H] bf16, dW1 [E, 2I, H] fp32, dW2 [E, H, I] fp32 after a
        forward with save_for_backward=True and prepare_backward_weights in the
        same mode.  x: the forward's BF16 input (high_precision only).
        ``mark(i)`` as in forward, over BACKWARD_STAGES."""
        if mode not in self.BACKWARD_MODES:
            raise ValueError(f"unknown backward mode {mode!r}")
        if getattr(self, "c1", None) is None:
            raise RuntimeError("backward needs a forward with save_for_backward=True")
        if getattr(self, "_w_mode", None) != mode:
            raise RuntimeError(f"prepare_backward_weights({mode!r}) first")
        if self.tile_m != 256:
            raise ValueError("the BF16 backward runs its GEMMs on CTA pairs: tile_m=256")
        if mode == "dequantized" and self.fc2 != "two_pass":
            raise ValueError("the dequantized backward reads the whole-row re-quantised D: "
                             "fc2='two_pass'")
        T, H, I, E, k, cap = self.T, self.H, self.I, self.E, self.k, self.cap
        seg, perm, inv, rp = self.seg
        mark = mark or (lambda i: None)
        bf = L.KIND_BF16
        mark(0)
        if mode == "high_precision":
            ops.moe_gather_bf16(x, perm, seg, E, k, cap, out=self.xp)
            d_op = self.d
        else:
            mv = seg[E:]
            ops.nvfp4_dequantize(*self.aq, 1, H, m_valid=mv, out=self.xp)
            ops.nvfp4_dequantize(*self.dq, 1, I, m_valid=mv, out=self.dop)
            d_op = self.dop
        return _bf16_backward_gemms(self, self.xp, d_op, self.w1_op, self.w2_op, dy, mark, 1)

    # kernels launched by one backward (weights prepared separately)
    LAUNCHES_PER_BACKWARD = {"high_precision": 7, "dequantized": 8}

    def backward_gemm_flops(self):
        """Algorithmic FLOPs of the four backward GEMMs over real rows."""
        R = self.T * self.k
        return 2 * (2 * R * self.H * 2 * self.I + 2 * R * self.I * self.H)

    def gemm_flops(self):
        """Algorithmic FLOPs of the two GEMMs over real (unpadded) rows:
        (FC1, FC2)."""
        R = self.T * self.k
        return 2 * R * self.H * 2 * self.I, 2 * R * self.I * self.H


# ============================================================================
# MXFP8
# ============================================================================

class MXFP8MoE:
    """Buffers and launch sequence of the MXFP8 expert layer, forward and
    backward, for a fixed (T, H, I, E, k).  tile_m as for NVFP4MoE; the wgrad
    GEMMs contract over the expert segments and run on CTA pairs too when the
    weight's row count is a multiple of 256."""

    def __init__(self, T, H, I, E, k, device="cuda", tile_m=256):
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.tile_m = tile_m
        dev = torch.device(device)
        cap = ops.moe_row_capacity(T, k, E, tile_m)
        self.cap = cap
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda *s, dtype: torch.empty(*s, dtype=dtype, device=dev)

        def mx(M, K, row=True, col=True):
            o = {}
            if row:
                o["row_q"] = e(M, K, dtype=u8)
                o["row_s"] = e(_sb(M, K // 32), dtype=u8)
            if col:
                o["col_q"] = e(K, M, dtype=u8)
                o["col_s"] = e(_sb(K, (M + 31) // 32), dtype=u8)
            return o

        self.seg = (e(E + 1, dtype=torch.int32), e(cap, dtype=torch.int32),
                    e(T * k, dtype=torch.int32), e(cap, dtype=f32))
        self.seg_ws = e(int(L.load().mpm_moe_segments_workspace_bytes(T, k, E)), dtype=u8)
        self.w1 = mx(E * 2 * I, H)
        self.w2 = mx(E * H, I)
        self.xp = e(cap, H, dtype=bf)
        self.xq = mx(cap, H)
        self.c1 = e(cap, 2 * I, dtype=bf)
        self.d = e(cap, I, dtype=bf)
        self.dq = mx(cap, I)
        self.y = e(cap, H, dtype=bf)
        self.out = e(T, H, dtype=bf)
        self.dyp = e(cap, H, dtype=bf)
        self.dyq = mx(cap, H)
        self.dh = e(cap, 2 * I, dtype=bf)
        self.dhq = mx(cap, 2 * I)
        self.dxp = e(cap, H, dtype=bf)
        self.dx = e(T, H, dtype=bf)
        self.dw1 = e(E, 2 * I, H, dtype=f32)
        self.dw2 = e(E, H, I, dtype=f32)

    # stages of one training step, for CUDA-event marks (see forward / backward)
    # (quant_x and quant_dy quantise the routed rows straight from the token
    # rows: the permute is folded into the quantiser's tile loads)
    STEP_STAGES = ("quant_w", "segments", "quant_x", "fc1", "quant_d", "fc2", "combine",
                   "quant_dy", "fc2_dgrad", "fc2_wgrad", "quant_dh", "fc1_dgrad", "combine_dx",
                   "fc1_wgrad")

    def quantize_weights(self, w1, w2):
        E, H, I = self.E, self.H, self.I
        ops.mxfp8_quantize(w1.reshape(E * 2 * I, H), ldc=E * 2 * I, out=self.w1)
        ops.mxfp8_quantize(w2.reshape(E * H, I), ldc=E * H, out=self.w2)

    def forward(self, x, topk_ids, topk_prob, mark=None):
        """``mark(i)`` (optional) before STEP_STAGES[i] for i = 1..6."""
        T, H, I, E, k, cap = self.T, self.H, self.I, self.E, self.k, self.cap
        mark = mark or (lambda i: None)
        seg, perm, inv, rp = self.seg
        mark(1)
        ops.moe_build_segments(topk_ids, topk_prob, E, out=self.seg, ws=self.seg_ws,
                               pad=self.tile_m)
        self._x = x                                  # for the high-precision BF16 backward
        mark(2)
        ops.mxfp8_quantize_gather(x, perm, seg, E, k, cap, ldc=cap, out=self.xq)
        mark(3)
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_SWIGLU_SAVE, E, cap, 2 * I, H, seg,
                             self.xq["row_q"], self.w1["row_q"], self.xq["row_s"], H // 32,
                             self.w1["row_s"], H // 32, self.c1, b_rows_per_expert=2 * I,
                             row_prob=rp, out2=self.d, tile_m=self.tile_m)
        mark(4)
        ops.mxfp8_quantize(self.d, ldc=cap, m_valid=seg[E:], out=self.dq)
        mark(5)
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, H, I, seg,
                             self.dq["row_q"], self.w2["row_q"], self.dq["row_s"], I // 32,
                             self.w2["row_s"], I // 32, self.y, b_rows_per_expert=H,
                             tile_m=self.tile_m)
        mark(6)
        ops.moe_combine(self.y, inv, T, k, out=self.out)
        return self.out

    def backward(self, dy, mark=None):
        """``mark(i)`` (optional) before STEP_STAGES[i] for i = 7..13 and once
        more (14) at the end."""
        T, H, I, E, k, cap = self.T, self.H, self.I, self.E, self.k, self.cap
        mark = mark or (lambda i: None)
        seg, perm, inv, rp = self.seg
        mark(7)
        ops.mxfp8_quantize_gather(dy, perm, seg, E, k, cap, ldc=cap, out=self.dyq)
        mark(8)
        # FC2 dgrad with the SwiGLU backward fused: dH = [dg | du]
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_DSWIGLU, E, cap, I, H, seg,
                             self.dyq["row_q"], self.w2["col_q"], self.dyq["row_s"], H // 32,
                             self.w2["col_s"], (E * H) // 32, self.dh, b_rows_per_expert=0,
                             b_k_per_expert=H, row_prob=rp, aux=self.c1, tile_m=self.tile_m)
        mark(9)
        # FC2 wgrad: dW2[e] = dY_e^T . D_e
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_K, L.EPI_F32, E, H, I, 0, seg,
                             self.dyq["col_q"], self.dq["col_q"], self.dyq["col_s"], cap // 32,
                             self.dq["col_s"], cap // 32, self.dw2, tile_m=self._wgrad_tile(H))
        mark(10)
        ops.mxfp8_quantize(self.dh, ldc=cap, m_valid=seg[E:], out=self.dhq)
        mark(11)
        # FC1 dgrad: dX_perm = dH . W1_e (column-wise W1 copy)
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_M, L.EPI_BF16, E, cap, H, 2 * I, seg,
                             self.dhq["row_q"], self.w1["col_q"], self.dhq["row_s"], (2 * I) // 32,
                             self.w1["col_s"], (E * 2 * I) // 32, self.dxp, b_rows_per_expert=0,
                             b_k_per_expert=2 * I, tile_m=self.tile_m)
        mark(12)
        ops.moe_combine(self.dxp, inv, T, k, out=self.dx)
        mark(13)
        # FC1 wgrad: dW1[e] = dH_e^T . X_e
        ops.moe_grouped_gemm(L.KIND_MXFP8, L.GROUP_K, L.EPI_F32, E, 2 * I, H, 0, seg,
                             self.dhq["col_q"], self.xq["col_q"], self.dhq["col_s"], cap // 32,
                             self.xq["col_s"], cap // 32, self.dw1, tile_m=self._wgrad_tile(2 * I))
        mark(14)
        return self.dx, self.dw1, self.dw2

    # ------------------------------------------------------------ BF16 backward
    # "The same backward mode selection applies to MXFP8": the four backward
    # GEMMs in BF16 on the original operands or on the BF16 dequantisation of
    # the row-wise MXFP8 copies the forward consumed.
    BACKWARD_MODES = ("high_precision", "dequantized")
    BF16_BACKWARD_STAGES = ("operands", "gather_dy", "fc2_dgrad", "fc2_wgrad", "fc1_dgrad",
                            "combine", "fc1_wgrad")

    def prepare_backward_weights(self, mode, w1=None, w2=None):
        """Weight operands of the BF16 dgrads, once per weight update: the
        BF16 weights (high_precision) or the dequantised row-wise MXFP8 copies
        made by quantize_weights (dequantized)."""
        E, H, I = self.E, self.H, self.I
        if mode == "high_precision":
            self.w1_op, self.w2_op = w1.reshape(E * 2 * I, H), w2.reshape(E * H, I)
        elif mode == "dequantized":
            self.w1_op = ops.mxfp8_dequantize(self.w1["row_q"], self.w1["row_s"])
            self.w2_op = ops.mxfp8_dequantize(self.w2["row_q"], self.w2["row_s"])
        else:
            raise ValueError(f"unknown backward mode {mode!r}")
        self._w_mode = mode

    def backward_bf16(self, dy, mode, mark=None):
        """dX, dW1, dW2 with BF16 GEMMs after forward(), in ``mode``
        (prepare_backward_weights first).  ``mark(i)`` over
        BF16_BACKWARD_STAGES."""
        if mode not in self.BACKWARD_MODES:
            raise ValueError(f"unknown backward mode {mode!r}")
        if getattr(self, "_w_mode", None) != mode:
            raise RuntimeError(f"prepare_backward_weights({mode!r}) first")
        if self.tile_m != 256:
            raise ValueError("the BF16 backward runs its GEMMs on CTA pairs: tile_m=256")
        H, I, E, cap = self.H, self.I, self.E, self.cap
        seg = self.seg[0]
        mark = mark or (lambda i: None)
        mark(0)
        if mode == "high_precision":
            # the forward quantised X straight from the token rows: the BF16
            # wgrad operand is gathered here
            ops.moe_gather_bf16(self._x, self.seg[1], seg, E, self.k, cap, out=self.xp)
            x_op, d_op = self.xp, self.d
        else:
            if getattr(self, "xop", None) is None:
                self.xop = torch.empty(cap, H, dtype=torch.bfloat16, device=self.xp.device)
                self.dop = torch.empty(cap, I, dtype=torch.bfloat16, device=self.xp.device)
            mv = seg[E:]
            ops.mxfp8_dequantize(self.xq["row_q"], self.xq["row_s"], m_valid=mv, out=self.xop)
            ops.mxfp8_dequantize(self.dq["row_q"], self.dq["row_s"], m_valid=mv, out=self.dop)
            x_op, d_op = self.xop, self.dop
        return _bf16_backward_gemms(self, x_op, d_op, self.w1_op, self.w2_op, dy, mark, 1)

    def _wgrad_tile(self, m_out):
        return 256 if (self.tile_m == 256 and m_out % 256 == 0) else 128

    def gemm_flops(self):
        R = self.T * self.k
        return 3 * (2 * R * self.H * 2 * self.I + 2 * R * self.I * self.H)
