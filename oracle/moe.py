"""MoE expert path: segments, permutation, grouped GEMMs, SwiGLU, combine.

Oracle: test infrastructure only.  All GEMMs run in fp64 on dequantised
codes (x_hat = q * s_b * s_g is exact in fp64), so the only rounding in a
GEMM result is the final rounding to the output dtype.

Sources: "miniTE technical report" section 5.2 (quantised outputs in one
contiguous buffer, expert boundaries given by offsets, zero-token experts and
padding handled in the same grouped path), section 5.3 (row amax accumulated
by the producer: the permute for FC1, the weighted SwiGLU for FC2), section
5.4 (FC1 epilogue: ACC x alpha_a[m] (x alpha_b), C = gate | up,
D = act(gate, up) x prob, amax of D), section 5.6 (single-pass FC2 fed tile
by tile with a running row amax and the partial sum rescaled when the outer
scale grows); "Towards Blackwell-native 8-bit and
4-bit RL", section "Recipe 1 / Training" (dgrad uses the column-wise weight
copy, wgrad the column-wise activation and gradient copies) and section
"High-precision and dequantized backward" (backward GEMMs in BF16 on the
original BF16 operands or on the BF16 dequantisation of the forward's
low-precision operands).

Readings the pages leave open (each one is fixed here):
* Segment order: rows of expert e are the (token, slot) pairs routed to e in
  ascending flat index t*k + j; each segment is padded to a multiple of 128
  rows; padding rows are all zero and carry probability 0.
* SwiGLU: D = silu(g) * u * p with g = FC1 output columns [0, I) and
  u = columns [I, 2I); silu(g) = g / (1 + exp(-g)).
* D is rounded to bf16 before its row amax and its re-quantisation.
* The FC2 output Y_perm is rounded to bf16; the combine sums each token's k
  rows in binary32, in slot order, and rounds the sum once to bf16.
* Backward: probabilities and routing are constants (no router gradient);
  dY_perm[row] = dY[token of row].
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import quant as Q

ROW_PAD = 128


def silu(g):
    return g / (1.0 + np.exp(-g))


def dsilu(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


# ------------------------------------------------------------ segments

def build_segments(topk_ids: np.ndarray, topk_prob: np.ndarray, E: int, pad=ROW_PAD):
    """Counting sort of the T*k routed (token, slot) pairs by expert.

    Returns seg_offsets int32 [E+1], perm int32 [R_pad] (flat index t*k + j,
    -1 for padding), inv_perm int32 [T*k] (flat index -> row), row_prob
    float32 [R_pad] (0 for padding).
    """
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    prob = np.asarray(topk_prob, dtype=np.float32).reshape(-1)
    counts = np.bincount(ids, minlength=E)
    padded = (counts + pad - 1) // pad * pad
    seg = np.zeros(E + 1, dtype=np.int64)
    seg[1:] = np.cumsum(padded)
    R_pad = int(seg[-1])
    perm = np.full(R_pad, -1, dtype=np.int64)
    inv = np.empty(ids.size, dtype=np.int64)
    fill = seg[:-1].copy()
    for f in range(ids.size):               # ascending flat index
        e = ids[f]
        inv[f] = fill[e]
        perm[fill[e]] = f
        fill[e] += 1
    row_prob = np.zeros(R_pad, dtype=np.float32)
    real = perm >= 0
    row_prob[real] = prob[perm[real]]
    return (seg.astype(np.int32), perm.astype(np.int32), inv.astype(np.int32),
            row_prob)


def expert_of_rows(seg_offsets: np.ndarray) -> np.ndarray:
    seg = np.asarray(seg_offsets, dtype=np.int64)
    e = np.repeat(np.arange(len(seg) - 1), np.diff(seg))
    return e


# ------------------------------------------------------------ grouped GEMM

def grouped_gemm(a: np.ndarray, b: np.ndarray, seg_offsets: np.ndarray) -> np.ndarray:
    """C[r, n] = sum_k a[r, k] * b[e(r), n, k] for the rows of each segment.

    a [R, K] fp64, b [E, N, K] fp64 -> C [R, N] fp64.  One library matmul per
    expert (the definition of a grouped GEMM, nothing more).
    """
    seg = np.asarray(seg_offsets, dtype=np.int64)
    R = a.shape[0]
    C = np.zeros((R, b.shape[1]), dtype=np.float64)
    for e in range(len(seg) - 1):
        r0, r1 = seg[e], seg[e + 1]
        if r1 > r0:
            C[r0:r1] = a[r0:r1] @ b[e].T
    return C


def grouped_wgrad(at: np.ndarray, bt: np.ndarray, seg_offsets: np.ndarray) -> np.ndarray:
    """dW[e] = at[:, seg e] @ bt[:, seg e].T : contraction over each expert's rows.

    at [N, R] fp64, bt [K, R] fp64 -> [E, N, K] fp64 (zero for empty experts).
    """
    seg = np.asarray(seg_offsets, dtype=np.int64)
    E = len(seg) - 1
    out = np.zeros((E, at.shape[0], bt.shape[0]), dtype=np.float64)
    for e in range(E):
        r0, r1 = seg[e], seg[e + 1]
        if r1 > r0:
            out[e] = at[:, r0:r1] @ bt[:, r0:r1].T
    return out


def gather_rows(x: np.ndarray, perm: np.ndarray, k: int) -> np.ndarray:
    """X_perm[row] = x[perm[row] // k]; zero rows for padding (perm = -1)."""
    perm = np.asarray(perm, dtype=np.int64)
    out = np.zeros((perm.size,) + x.shape[1:], dtype=x.dtype)
    real = perm >= 0
    out[real] = x[perm[real] // k]
    return out


def combine(y_perm: np.ndarray, inv_perm: np.ndarray, T: int, k: int) -> np.ndarray:
    """out[t] = bf16( y[inv[t*k]] + y[inv[t*k + 1]] + ... + y[inv[t*k + k-1]] ).

    "miniTE technical report", section 5.3: each token's output is the sum of
    its k expert outputs (the router weight was already applied to D in the
    FC1 epilogue).  The section gives no accumulation order or precision, so
    the reading fixed here is: start from +0.0 in binary32, add the token's
    rows one at a time in slot order j = 0 .. k-1, each addition one IEEE
    binary32 round-to-nearest-even step (numpy float32 arithmetic), then
    round the binary32 sum once to bf16 (nearest, ties to even).  The order
    matters: an fp64 sum, or another slot order, can land on another bf16
    value.  y_perm holds bf16 values (exact in binary32).  Returns the bf16
    values as fp64.
    """
    y = np.asarray(y_perm)
    y32 = y.astype(np.float32)
    assert np.array_equal(y32.astype(y.dtype), y), "combine input must be exact in binary32"
    inv = np.asarray(inv_perm, dtype=np.int64).reshape(T, k)
    acc = np.zeros((T,) + y.shape[1:], dtype=np.float32)
    for j in range(k):
        acc = np.add(acc, y32[inv[:, j]], dtype=np.float32)
    return F.bf16_bits_to_f32(F.f32_to_bf16_bits(acc)).astype(np.float64)


# ------------------------------------------------------------ NVFP4 forward

def nvfp4_weights(w1: np.ndarray, w2: np.ndarray):
    """Quantise W1 [E, 2I, H] (gate|up jointly) and W2 [E, H, I] per expert."""
    E, I2, H = w1.shape
    I = I2 // 2
    w1q = Q.nvfp4_quantize_joint([w1[:, :I], w1[:, I:]], E)
    w2q = Q.nvfp4_quantize_joint([w2], E)
    return w1q, w2q


def dequant_weights_nvfp4(wq):
    packed, sb, sg = wq
    E, R, _ = packed.shape
    return np.stack([Q.nvfp4_dequantize(packed[e], sb[e], sg[e]) for e in range(E)])


def fc1_epilogue(acc: np.ndarray, row_prob: np.ndarray, I: int) -> np.ndarray:
    """D = bf16( silu(g) * u * p ); acc already carries alpha_a * alpha_b."""
    g, u = acc[:, :I], acc[:, I:2 * I]
    d = silu(g) * u * np.asarray(row_prob, dtype=np.float64)[:, None]
    return F.bf16_round(d)


def nvfp4_moe_forward(x: np.ndarray, topk_ids, topk_prob, w1, w2, E: int, pad=ROW_PAD):
    """The full NVFP4 expert-layer forward.

    x [T, H] bf16 values; w1 [E, 2I, H]; w2 [E, H, I].  Returns a dict with
    every intermediate the CUDA path materialises (in the permuted layout with
    segments padded to ``pad`` rows; the padding changes the layout only).
    """
    T, H = x.shape
    k = np.asarray(topk_ids).shape[1]
    I = w1.shape[1] // 2
    # per-token activation quantisation of X (once per token)
    qx, sx, tsx = Q.nvfp4_quantize_per_token(x)
    seg, perm, inv, row_prob = build_segments(topk_ids, topk_prob, E, pad)
    xq_deq = Q.nvfp4_dequantize(qx, sx, tsx)                 # [T, H]
    a1 = gather_rows(xq_deq, perm, k)                        # [R_pad, H]
    (w1p, w1s, w1g), (w2p, w2s, w2g) = nvfp4_weights(w1, w2)
    b1 = dequant_weights_nvfp4((w1p, w1s, w1g))
    acc1 = grouped_gemm(a1, b1, seg)                         # fp64
    d = fc1_epilogue(acc1, row_prob, I)
    amax_d = np.max(np.abs(d), axis=1).astype(np.float32)
    qd, sd, tsd = Q.nvfp4_quantize_per_token(d, amax_d)
    b2 = dequant_weights_nvfp4((w2p, w2s, w2g))
    y = grouped_gemm(Q.nvfp4_dequantize(qd, sd, tsd), b2, seg)
    y_bf16 = F.bf16_round(y)
    out = combine(y_bf16, inv, T, k)
    return dict(qx=qx, sx=sx, tsx=tsx, seg=seg, perm=perm, inv=inv,
                row_prob=row_prob, w1=(w1p, w1s, w1g), w2=(w2p, w2s, w2g),
                acc1=acc1, d=d, amax_d=amax_d, qd=qd, sd=sd, tsd=tsd,
                y=y_bf16, out=out)


def nvfp4_fc2_online_amax(d: np.ndarray, seg_offsets: np.ndarray, w2q, tile_k: int = 256):
    """FC2 of the single-pass fused FFN with online amax compensation
    ("miniTE technical report", section 5.6).

    The fused path never holds a whole row of D before FC2 consumes it: FC2
    walks its K dimension (= I) in tiles P_i of ``tile_k`` columns as FC1 and
    SwiGLU produce them.  Per row, in tile order:

      gamax <- max(gamax, max|P_i|)      the running row amax
      gs     = gamax / 2688             the per-token outer-scale rule
      (s_b, q) = NVFP4 block encoding of P_i against gs (blocks of 16)
      dO_i   = (q s_b) (q_W s_bW)^T      block scales applied, neither gs nor
                                         the weight's tensor scale
      O      = O * (gs_prev / gs) + dO_i,  gs_prev = gs

    A row whose gamax is still 0 skips the tile (its contribution so far is
    zero); at the end Y = O * gs_prev * s_g(W2_e), and an all-zero row gives 0.

    Readings the section leaves open (each fixed here): P_i is the tile of
    the weighted SwiGLU output rounded to bf16, i.e. the values the two-pass
    path writes as D; gs, s_b and q follow the canonical fp32 sequence of the
    per-token quantiser (with its 2**-116 floor) with gs in place of s_g; the
    last tile may be shorter than ``tile_k`` (any multiple of 16); O and the
    ratio gs_prev / gs are carried in fp64 and Y is rounded once to bf16.

    d [R_pad, I] in the permuted layout; w2q = (packed [E, H, I/2], block
    scales [E, H, I/16], s_g [E]).  Returns y (bf16 values) and y64 (before
    rounding) [R_pad, H], the per-tile codes [R_pad, I] and block scales
    [R_pad, I/16] the fused path would feed to FC2 (never materialised
    there), and gs [R_pad, n_tiles].
    """
    d = np.asarray(d, dtype=np.float32)
    R, I = d.shape
    w2p, w2s, w2g = w2q
    E, H, _ = w2p.shape
    assert tile_k > 0 and tile_k % Q.NV_BLOCK == 0 and I % Q.NV_BLOCK == 0
    tiles = [(c0, min(c0 + tile_k, I)) for c0 in range(0, I, tile_k)]
    codes = np.zeros((R, I), dtype=np.uint8)
    sb = np.zeros((R, I // Q.NV_BLOCK), dtype=np.uint8)
    gs_tiles = np.zeros((R, len(tiles)), dtype=np.float32)
    y64 = np.zeros((R, H))
    for e in range(E):
        r0, r1 = int(seg_offsets[e]), int(seg_offsets[e + 1])
        if r1 == r0:
            continue
        bw = Q.nvfp4_dequantize(w2p[e], w2s[e], 1.0)         # q_W * s_bW, [H, I]
        gamax = np.zeros(r1 - r0, dtype=np.float32)
        gs_prev = np.zeros(r1 - r0, dtype=np.float32)
        o = np.zeros((r1 - r0, H))
        for i, (c0, c1) in enumerate(tiles):
            p = d[r0:r1, c0:c1]
            gamax = np.maximum(gamax, np.max(np.abs(p), axis=1))
            live = gamax > 0
            gs = Q.nvfp4_outer_scale(gamax)
            q, s = Q.nvfp4_encode_with_outer(p, gs)
            xs = F.e2m1_decode(q) * np.repeat(F.e4m3_decode(s), Q.NV_BLOCK, axis=1)
            do = xs @ bw[:, c0:c1].T
            ratio = np.zeros(r1 - r0)
            np.divide(gs_prev.astype(np.float64), gs.astype(np.float64), out=ratio, where=live)
            o = np.where(live[:, None], o * ratio[:, None] + do, o)
            gs_prev = np.where(live, gs, gs_prev)
            codes[r0:r1, c0:c1] = q
            sb[r0:r1, c0 // Q.NV_BLOCK:c1 // Q.NV_BLOCK] = s
            gs_tiles[r0:r1, i] = gs
        y64[r0:r1] = o * gs_prev.astype(np.float64)[:, None] * float(w2g[e])
    return dict(y=F.bf16_round(y64), y64=y64, codes=codes, sb=sb, gs=gs_tiles)


def nvfp4_moe_forward_single_pass(x: np.ndarray, topk_ids, topk_prob, w1, w2, E: int,
                                  tile_k: int = 256, pad=ROW_PAD):
    """The NVFP4 expert layer with FC2 fed tile by tile (section 5.6 of the
    miniTE report): the same quantised X, segments, FC1 and SwiGLU as the
    two-pass forward, then ``nvfp4_fc2_online_amax`` on D instead of the
    whole-row re-quantisation, then the combine.  Returns the online FC2's
    outputs, the layer output and the two-pass forward's dict (``two_pass``)."""
    T = x.shape[0]
    k = np.asarray(topk_ids).shape[1]
    r = nvfp4_moe_forward(x, topk_ids, topk_prob, w1, w2, E, pad)
    s = nvfp4_fc2_online_amax(r["d"], r["seg"], r["w2"], tile_k)
    s["out"] = combine(s["y"], r["inv"], T, k)
    s["two_pass"] = r
    return s


def nvfp4_gemm_single(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray):
    """One expert, no SwiGLU: per-token X quantisation, joint gate/up weight
    quantisation, C = deq(X) deq(W)^T in fp64 ([M, 2N], fp32 output)."""
    qx, sx, tsx = Q.nvfp4_quantize_per_token(x)
    wp, ws, wg = Q.nvfp4_quantize_joint([w_gate[None], w_up[None]], 1)
    a = Q.nvfp4_dequantize(qx, sx, tsx)
    b = Q.nvfp4_dequantize(wp[0], ws[0], wg[0])
    c = a @ b.T
    return dict(qx=qx, sx=sx, tsx=tsx, wq=(wp, ws, wg), c=c)


# ------------------------------------------------------------ MXFP8 fwd + bwd

def mx_rows(x):
    """Row-wise MXFP8 round trip: dequantised fp64 values [R, C]."""
    c, s = Q.mxfp8_quantize_rowwise(x)
    return Q.mxfp8_dequantize(c, s)


def mx_cols_t(x):
    """Column-wise MXFP8 copy, dequantised, in its stored transposed form [C, R]."""
    c, s = Q.mxfp8_quantize_colwise(x)
    return Q.mxfp8_dequantize(c, s)


def swiglu_backward(dd: np.ndarray, c1: np.ndarray, row_prob: np.ndarray, I: int):
    """dH = [dg | du] for D = silu(g) * u * p (p constant)."""
    g, u = c1[:, :I], c1[:, I:2 * I]
    p = np.asarray(row_prob, dtype=np.float64)[:, None]
    dg = dd * p * u * dsilu(g)
    du = dd * p * silu(g)
    return np.concatenate([dg, du], axis=1)


def mxfp8_moe_fwd_bwd(x, topk_ids, topk_prob, w1, w2, dy, E: int, pad=ROW_PAD):
    """End-to-end MXFP8 expert layer, forward and backward.

    Every GEMM operand is quantised from bf16: fprop uses row-wise copies,
    dgrad the row-wise gradient and the column-wise weight, wgrad the
    column-wise gradient and activation copies.
    """
    T, H = x.shape
    k = np.asarray(topk_ids).shape[1]
    I = w1.shape[1] // 2
    seg, perm, inv, row_prob = build_segments(topk_ids, topk_prob, E, pad)
    xp = gather_rows(np.asarray(x, dtype=np.float64), perm, k)     # bf16 values
    # forward FC1
    b1 = np.stack([mx_rows(w1[e]) for e in range(E)])              # [E, 2I, H]
    acc1 = grouped_gemm(mx_rows(xp), b1, seg)
    c1 = F.bf16_round(acc1)                                        # saved gate|up
    d = fc1_epilogue(acc1, row_prob, I)
    # forward FC2
    b2 = np.stack([mx_rows(w2[e]) for e in range(E)])              # [E, H, I]
    y = F.bf16_round(grouped_gemm(mx_rows(d), b2, seg))
    out = combine(y, inv, T, k)
    # backward
    dyp = gather_rows(np.asarray(dy, dtype=np.float64), perm, k)   # [R_pad, H]
    w2c = np.stack([mx_cols_t(w2[e]) for e in range(E)])           # [E, I, H]
    dd = grouped_gemm(mx_rows(dyp), w2c, seg)                      # [R_pad, I] fp64
    dw2 = grouped_wgrad(mx_cols_t(dyp), mx_cols_t(d), seg)         # [E, H, I]
    dh = F.bf16_round(swiglu_backward(dd, c1, row_prob, I))        # [R_pad, 2I]
    w1c = np.stack([mx_cols_t(w1[e]) for e in range(E)])           # [E, H, 2I]
    dxp = F.bf16_round(grouped_gemm(mx_rows(dh), w1c, seg))        # [R_pad, H]
    dx = combine(dxp, inv, T, k)
    dw1 = grouped_wgrad(mx_cols_t(dh), mx_cols_t(xp), seg)         # [E, 2I, H]
    return dict(seg=seg, perm=perm, inv=inv, row_prob=row_prob, c1=c1, d=d,
                y=y, out=out, dd=dd, dh=dh, dxp=dxp, dx=dx, dw1=dw1, dw2=dw2)


# ------------------------------------------------------------ BF16 backward

BACKWARD_MODES = ("high_precision", "dequantized")


def bf16_backward(xp, w1, w2, d, c1, dyp, seg, row_prob, I: int):
    """Backward of the expert FFN with BF16 GEMMs on the given operands.

    xp [R, H], w1 [E, 2I, H], w2 [E, H, I], d [R, I] (the FC2 input),
    c1 [R, 2I] (the FC1 output gate|up, where the SwiGLU derivative is
    taken), dyp [R, H]: the permuted output gradient.  GEMMs in fp64 (one
    library matmul per expert); dH and dX_perm rounded to bf16 as the kernels
    store them, dW1 / dW2 left in fp64 (the kernels store fp32).

      dD      = dY_perm W2_e                 [R, I]
      dH      = SwiGLU'(C1; dD, p)           [R, 2I]
      dX_perm = dH W1_e                      [R, H]
      dW2_e   = dY_perm_e^T D_e              [H, I]
      dW1_e   = dH_e^T X_perm_e              [2I, H]
    """
    w2t = np.transpose(np.asarray(w2, dtype=np.float64), (0, 2, 1))     # [E, I, H]
    w1t = np.transpose(np.asarray(w1, dtype=np.float64), (0, 2, 1))     # [E, H, 2I]
    dd = grouped_gemm(dyp, w2t, seg)
    dh = F.bf16_round(swiglu_backward(dd, c1, row_prob, I))
    dxp = F.bf16_round(grouped_gemm(dh, w1t, seg))
    dw2 = grouped_wgrad(np.asarray(dyp).T, np.asarray(d).T, seg)
    dw1 = grouped_wgrad(dh.T, np.asarray(xp).T, seg)
    return dict(dd=dd, dh=dh, dxp=dxp, dw1=dw1, dw2=dw2)


def nvfp4_backward_operands(fwd: dict, x, w1, w2, mode: str):
    """(X_perm, W1, W2, D) of the BF16 backward after an NVFP4 forward.

    high_precision: the original BF16 operands (X gathered by expert, the
    BF16 weights, the BF16 D the FC1 epilogue produced before its
    re-quantisation).  dequantized: the BF16 dequantisation of exactly the
    NVFP4 operands the forward GEMMs consumed (per-token X codes, the jointly
    scaled W1 codes, W2 codes, the re-quantised D codes).
    """
    k = int(np.asarray(fwd["inv"]).size // np.asarray(x).shape[0])
    perm = fwd["perm"]
    if mode == "high_precision":
        xp = gather_rows(np.asarray(x, dtype=np.float64), perm, k)
        return xp, np.asarray(w1, np.float64), np.asarray(w2, np.float64), fwd["d"]
    if mode == "dequantized":
        xq = Q.nvfp4_dequantize_bf16(fwd["qx"], fwd["sx"], fwd["tsx"])
        xp = gather_rows(xq, perm, k)
        (w1p, w1s, w1g), (w2p, w2s, w2g) = fwd["w1"], fwd["w2"]
        E = w1p.shape[0]
        b1 = np.stack([Q.nvfp4_dequantize_bf16(w1p[e], w1s[e], w1g[e]) for e in range(E)])
        b2 = np.stack([Q.nvfp4_dequantize_bf16(w2p[e], w2s[e], w2g[e]) for e in range(E)])
        dhat = Q.nvfp4_dequantize_bf16(fwd["qd"], fwd["sd"], fwd["tsd"])
        return xp, b1, b2, dhat
    raise ValueError(f"unknown backward mode {mode!r}")


def nvfp4_moe_backward_bf16(fwd: dict, x, w1, w2, dy, mode: str):
    """BF16 backward of the NVFP4 expert layer (``fwd`` from nvfp4_moe_forward).

    The SwiGLU derivative is taken at the forward's own FC1 output C1 (the
    fp64 GEMM of the NVFP4 operands, rounded to bf16 as the forward saves
    it); routing and probabilities are constants.  Returns the dict of
    bf16_backward plus dx = combine(dX_perm) and the operands used.
    """
    T = np.asarray(x).shape[0]
    inv = np.asarray(fwd["inv"])
    k = inv.size // T
    I = np.asarray(w1).shape[1] // 2
    xp, b1, b2, d = nvfp4_backward_operands(fwd, x, w1, w2, mode)
    c1 = F.bf16_round(fwd["acc1"])
    dyp = gather_rows(np.asarray(dy, dtype=np.float64), fwd["perm"], k)
    r = bf16_backward(xp, b1, b2, d, c1, dyp, fwd["seg"], fwd["row_prob"], I)
    r["dx"] = combine(r["dxp"], inv, T, k)
    r.update(xp=xp, w1_op=b1, w2_op=b2, d_op=d, c1=c1, dyp=dyp)
    return r


def mxfp8_moe_bf16_backward(x, topk_ids, topk_prob, w1, w2, dy, E: int, mode: str, pad=ROW_PAD):
    """MXFP8 forward (row-wise copies, as in mxfp8_moe_fwd_bwd) followed by
    the BF16 backward in one of the two operand modes: high_precision uses
    the BF16 X_perm, W1, W2 and the FC1 epilogue's BF16 D; dequantized uses
    the BF16 dequantisation of the row-wise MXFP8 copies the forward GEMMs
    consumed (X_perm, W1, W2, D).  The SwiGLU derivative is taken at the
    saved C = gate|up (bf16)."""
    T, H = np.asarray(x).shape
    k = np.asarray(topk_ids).shape[1]
    I = np.asarray(w1).shape[1] // 2
    seg, perm, inv, row_prob = build_segments(topk_ids, topk_prob, E, pad)
    xp = gather_rows(np.asarray(x, dtype=np.float64), perm, k)
    b1 = np.stack([mx_rows(w1[e]) for e in range(E)])
    acc1 = grouped_gemm(mx_rows(xp), b1, seg)
    c1 = F.bf16_round(acc1)
    d = fc1_epilogue(acc1, row_prob, I)
    if mode == "high_precision":
        x_op, w1_op, w2_op, d_op = xp, np.asarray(w1, np.float64), np.asarray(w2, np.float64), d
    elif mode == "dequantized":
        x_op = F.bf16_round(mx_rows(xp))
        w1_op = F.bf16_round(b1)
        w2_op = F.bf16_round(np.stack([mx_rows(w2[e]) for e in range(E)]))
        d_op = F.bf16_round(mx_rows(d))
    else:
        raise ValueError(f"unknown backward mode {mode!r}")
    dyp = gather_rows(np.asarray(dy, dtype=np.float64), perm, k)
    r = bf16_backward(x_op, w1_op, w2_op, d_op, c1, dyp, seg, row_prob, I)
    r["dx"] = combine(r["dxp"], inv, T, k)
    r.update(seg=seg, perm=perm, inv=inv, row_prob=row_prob, c1=c1, d=d, xp=x_op,
             w1_op=w1_op, w2_op=w2_op, d_op=d_op, dyp=dyp)
    return r
