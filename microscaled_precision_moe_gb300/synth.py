"""Seeded, counter-based synthetic inputs shared by the CUDA path and the oracle.

This module holds input generation only: none of the quantisation, GEMM or
routing-kernel arithmetic lives here. Every element is a pure function of
(seed, tensor id, flat index), so any slice of any tensor can be regenerated on
its own, on the host or on a device, without materialising the rest.

Definition (one counter-based generator, written out so that each side can
re-implement it):

* ``key(seed, tensor_id) = splitmix64_mix(seed * 0x100000001B3 + tensor_id)``
  (python integers, modulo 2**64).
* ``word(key, i) = splitmix64_mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` -- the
  i-th output of a splitmix64 stream started at ``key``.
* ``unif(key, i) = (word >> 11) * 2**-53`` in [0, 1).
* A normal draw for element j uses words 3j and 3j+1 (Box-Muller in fp64,
  cosine branch); word 3j+2 decides an outlier (``unif < p`` multiplies the
  value by the outlier factor).
* The fp64 value is rounded to fp32 (round-to-nearest-even) and then to bf16
  (round-to-nearest-even).

All arithmetic runs in torch on the requested device, int64 with
two's-complement wrap-around for the 64-bit mixing.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

_M64 = (1 << 64) - 1


def _s64(c: int) -> int:
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MIX1 = _s64(0xBF58476D1CE4E5B9)
_MIX2 = _s64(0x94D049BB133111EB)


def _mix_py(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_py(key: int, i: int) -> int:
    """Pure-python reference of ``word(key, i)`` (unsigned)."""
    return _mix_py((key + (i + 1) * 0x9E3779B97F4A7C15) & _M64)


def stream_key(seed: int, tensor_id: int) -> int:
    return _mix_py(seed * 0x100000001B3 + tensor_id)


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    # logical right shift of int64 bit patterns
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _MIX1
    z = (z ^ _srl(z, 27)) * _MIX2
    return z ^ _srl(z, 31)


def words(key: int, idx: torch.Tensor) -> torch.Tensor:
    """int64 bit patterns of word(key, idx) for an int64 index tensor."""
    return _mix(_s64(key) + (idx + 1) * _GOLDEN)


def unif(key: int, idx: torch.Tensor) -> torch.Tensor:
    return _srl(words(key, idx), 11).to(torch.float64) * (2.0 ** -53)


def unif_open(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Uniform in the open interval (0, 1)."""
    return (_srl(words(key, idx), 11).to(torch.float64) + 0.5) * (2.0 ** -53)


def normal_f64(key: int, start: int, count: int, device="cpu",
               std: float = 1.0, outlier_p: float = 0.0,
               outlier_mul: float = 1.0) -> torch.Tensor:
    """fp64 draws for flat elements [start, start+count) of one tensor."""
    j = torch.arange(start, start + count, dtype=torch.int64, device=device)
    u1 = unif(key, 3 * j)
    u2 = unif(key, 3 * j + 1)
    z = torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2)
    z = z * std
    if outlier_p > 0.0:
        u3 = unif(key, 3 * j + 2)
        z = torch.where(u3 < outlier_p, z * outlier_mul, z)
    return z


def to_bf16(x64: torch.Tensor) -> torch.Tensor:
    return x64.to(torch.float32).to(torch.bfloat16)


def normal_bf16(seed: int, tensor_id: int, shape, device="cpu", std=1.0,
                outlier_p=0.0, outlier_mul=1.0, chunk=1 << 26) -> torch.Tensor:
    """A bf16 tensor of the given shape, generated in chunks of flat elements."""
    n = 1
    for s in shape:
        n *= int(s)
    key = stream_key(seed, tensor_id)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s0 in range(0, n, chunk):
        c = min(chunk, n - s0)
        out[s0:s0 + c] = to_bf16(normal_f64(key, s0, c, device, std,
                                            outlier_p, outlier_mul))
    return out.view(*shape)


def normal_bf16_rows(seed: int, tensor_id: int, ncols: int, rows: torch.Tensor,
                     device="cpu", std=1.0, outlier_p=0.0,
                     outlier_mul=1.0) -> torch.Tensor:
    """Selected rows of a row-major [*, ncols] tensor from ``normal_bf16``."""
    key = stream_key(seed, tensor_id)
    rows = rows.to(torch.int64).to(device)
    j = (rows[:, None] * ncols
         + torch.arange(ncols, dtype=torch.int64, device=device)[None, :]).reshape(-1)
    u1 = unif(key, 3 * j)
    u2 = unif(key, 3 * j + 1)
    z = torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2) * std
    if outlier_p > 0.0:
        u3 = unif(key, 3 * j + 2)
        z = torch.where(u3 < outlier_p, z * outlier_mul, z)
    return to_bf16(z).view(rows.numel(), ncols)


# --------------------------------------------------------------------------
# Tensor ids (one stream per logical tensor)
# --------------------------------------------------------------------------
TID_X = 1
TID_WGATE = 2
TID_WUP = 3
TID_W1 = 4
TID_W2 = 5
TID_LOGITS = 6
TID_DY = 7
TID_ROWSCALE = 8
TID_SPECIAL = 9


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int        # tokens
    H: int        # hidden
    I: int        # expert intermediate
    E: int        # experts
    k: int = 8    # top-k
    w_std: float = 0.02
    w_outlier_p: float = 0.0
    w_outlier_mul: float = 1.0
    zipf: float = 0.0   # 0 => softmax over N(0,1) logits, else Zipf(zipf) Gumbel-top-k


# NVFP4 forward, 30B-A3B-like layer
MOE_30B = MoEShape("nvfp4_moe_fwd_T16384_H2048_I768_E128_k8", 16384, 2048, 768, 128)
# MXFP8 forward+backward, same layer, 8192 tokens
MOE_30B_BWD = MoEShape("mxfp8_moe_fwdbwd_T8192_H2048_I768_E128_k8", 8192, 2048, 768, 128)
# NVFP4 forward, 671B-like layer with Zipf(1.1) expert load
MOE_671B = MoEShape("nvfp4_moe_fwd_T32768_H7168_I2048_E256_k8_zipf1.1", 32768, 7168,
                    2048, 256, w_std=0.01, w_outlier_p=1e-4, w_outlier_mul=100.0,
                    zipf=1.1)


def scaled(shape: MoEShape, T=None, H=None, I=None, E=None, k=None,
           name=None) -> MoEShape:
    """A reduced copy of a workload (same distributions, smaller sizes)."""
    E = E or shape.E
    k = k or min(shape.k, E)
    return MoEShape(name or (shape.name + "_small"), T or shape.T, H or shape.H,
                    I or shape.I, E, k, shape.w_std,
                    shape.w_outlier_p, shape.w_outlier_mul, shape.zipf)


# --------------------------------------------------------------------------
# Single-expert gate/up (128 x 2048 activations, 768 x 2048 gate and up)
# --------------------------------------------------------------------------
def single_expert_inputs(seed=0, M=128, K=2048, N_half=768, device="cpu"):
    x = normal_bf16(seed, TID_X, (M, K), device, 1.0, 1e-3, 50.0)
    wg = normal_bf16(seed, TID_WGATE, (N_half, K), device, 0.02)
    wu = normal_bf16(seed, TID_WUP, (N_half, K), device, 0.02)
    return x, wg, wu


# --------------------------------------------------------------------------
# MXFP8 quantiser input: N(0,1) rows, 1% of rows x1e3, then 32 zero rows,
# 32 rows of +-448 and 32 rows of random bf16 subnormals
# --------------------------------------------------------------------------
def mxfp8_quantizer_input(seed=0, M=8192, K=2048, device="cpu"):
    body = normal_f64(stream_key(seed, TID_X), 0, M * K, device).view(M, K)
    rkey = stream_key(seed, TID_ROWSCALE)
    big = unif(rkey, torch.arange(M, dtype=torch.int64, device=device)) < 0.01
    body = torch.where(big[:, None], body * 1e3, body)
    body = to_bf16(body)
    skey = stream_key(seed, TID_SPECIAL)
    zeros = torch.zeros(32, K, dtype=torch.bfloat16, device=device)
    idx = torch.arange(32 * K, dtype=torch.int64, device=device)
    sgn = torch.where(unif(skey, idx) < 0.5, -1.0, 1.0)
    maxes = (448.0 * sgn).view(32, K).to(torch.bfloat16)
    # subnormal bf16 bit patterns 0x0001..0x007F with a random sign
    mag = (_srl(words(skey, idx + 32 * K), 40) % 127 + 1)
    neg = unif(skey, idx + 64 * K) < 0.5
    bits = torch.where(neg, mag | 0x8000, mag).to(torch.int32)
    bits = torch.where(bits >= 0x8000, bits - 0x10000, bits).to(torch.int16)
    subn = bits.view(torch.bfloat16).view(32, K)
    return torch.cat([body, zeros, maxes, subn], dim=0)


# --------------------------------------------------------------------------
# Routing inputs (prepared once on the host, shared by both sides)
# --------------------------------------------------------------------------
def routing(shape: MoEShape, seed=0):
    """topk_ids int32 [T,k] and topk_prob fp32 [T,k].

    Without Zipf skew: logits ~ N(0,1), softmax over the E experts, top-k with
    ties to the lower expert id, the k probabilities renormalised to sum to 1.
    With Zipf skew s: logit[t,e] = log p_e + Gumbel(0,1), p_e ~ (e+1)^-s; the
    top-k of the perturbed logits are k distinct experts drawn with
    probability ~ p_e; the gate weights are the softmax of those k logits.
    """
    T, E, k = shape.T, shape.E, shape.k
    key = stream_key(seed, TID_LOGITS)
    if shape.zipf == 0.0:
        logits = normal_f64(key, 0, T * E).view(T, E)
    else:
        e = torch.arange(E, dtype=torch.float64)
        p = (e + 1.0) ** (-shape.zipf)
        p = p / p.sum()
        u = unif_open(key, torch.arange(T * E, dtype=torch.int64)).view(T, E)
        logits = torch.log(p)[None, :] - torch.log(-torch.log(u))
    order = torch.sort(-logits, dim=1, stable=True).indices[:, :k]
    sel = torch.gather(logits, 1, order)
    if shape.zipf == 0.0:
        full = torch.softmax(logits, dim=1)
        pr = torch.gather(full, 1, order)
        pr = pr / pr.sum(dim=1, keepdim=True)
    else:
        pr = torch.softmax(sel, dim=1)
    return order.to(torch.int32).contiguous(), pr.to(torch.float32).contiguous()


def moe_activations(shape: MoEShape, seed=0, device="cpu", rows=None):
    """X [T,H] bf16 ~ N(0,1) (all rows, or only ``rows``)."""
    if rows is None:
        return normal_bf16(seed, TID_X, (shape.T, shape.H), device)
    return normal_bf16_rows(seed, TID_X, shape.H, rows, device)


def moe_weights(shape: MoEShape, seed=0, device="cpu", experts=None):
    """W1 [E,2I,H] (gate rows [0,I), up rows [I,2I)) and W2 [E,H,I], bf16.

    ``experts`` selects a subset (the returned tensors then hold only those
    experts, in the given order); each expert's elements are the same as in the
    full tensor.
    """
    E, H, I = shape.E, shape.H, shape.I
    kw = dict(std=shape.w_std, outlier_p=shape.w_outlier_p,
              outlier_mul=shape.w_outlier_mul)
    if experts is None:
        w1 = normal_bf16(seed, TID_W1, (E, 2 * I, H), device, **kw)
        w2 = normal_bf16(seed, TID_W2, (E, H, I), device, **kw)
        return w1, w2
    k1, k2 = stream_key(seed, TID_W1), stream_key(seed, TID_W2)
    w1s, w2s = [], []
    for e in experts:
        n1 = 2 * I * H
        w1s.append(to_bf16(normal_f64(k1, int(e) * n1, n1, device, **kw)).view(2 * I, H))
        n2 = H * I
        w2s.append(to_bf16(normal_f64(k2, int(e) * n2, n2, device, **kw)).view(H, I))
    return torch.stack(w1s), torch.stack(w2s)


def moe_grad_out(shape: MoEShape, seed=0, device="cpu"):
    """dY [T,H] bf16 ~ N(0, 1e-3)."""
    return normal_bf16(seed, TID_DY, (shape.T, shape.H), device, std=1e-3)
