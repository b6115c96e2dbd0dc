#!/usr/bin/env python3
"""Benchmark of the microscaled-precision MoE hot path on one GB300.

Headline step: one NVFP4 expert-layer forward of the 671B-shaped layer
(32768 tokens, hidden 7168, 256 experts, intermediate 2048, top-8 with
Zipf(1.1) expert load): per-token activation quantisation, segment build,
gather, FC1 grouped GEMM + SwiGLU x prob + row amax, re-quantisation reusing
the amax, FC2 grouped GEMM, combine.  Weights are quantised once, outside the
step (a weight update is a separate event), and timed separately.

value = algorithmic GEMM FLOPs of the step (real rows, padding excluded) /
step time, in TFLOP/s.  Inputs are resident in HBM and larger than L2
(activations 470 MB, FP4 weights 5.6 GB), so no L2 flush is needed.
Secondary lines (same JSON, key "also"): quantiser GB/s against HBM, the MXFP8
layer forward+backward on the 30B-shaped layer, the NVFP4 30B-shaped forward,
the BF16 (high-precision and dequantized) backward of the NVFP4 layer,
decode-sized batches of the 671B-shaped layer on the small-M kernel, and the
single-expert NVFP4 GEMM (128 x 2048 activations against 1536 x 2048 gate|up
weights) with its activation quantisation, each timed separately.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantizer HBM GB/s; NVFP4/MXFP8 grouped-GEMM TFLOPS; % of GB300 roofline"
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25      # dense nominal ratio (B300 row of the pages)
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------- distributed

def _dist(backend=None):
    """(torch.distributed or None, rank, world) from the torchrun environment;
    one replica per GPU over NCCL, or gloo when no GPU is present."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, ws
    return None, 0, 1


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, v: float) -> float:
    """The slowest replica's time (every rank gets it)."""
    if dist is None:
        return v
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) during the timed region.  nvidia-smi
    takes longer to start than a short timed region lasts, so entering waits
    (at most 3 s) for its first sample, and the summary keeps only the
    samples that arrived after that (all of them if none did)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.first = 0
        self._ready = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            self._ready.wait(timeout=3.0)
            self.first = len(self.lines)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self._ready.set()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = self.lines[self.first:] if len(self.lines) > self.first else self.lines
        for l in inside:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle CPU arm

def _oracle_prepare(shape, ids, prob, n_experts=1, seed=0):
    """Inputs of a bounded CPU sample of the workload: the whole routed row
    set of n_experts experts of median load (their bf16 activations, their
    bf16 W1 and W2, the router weights)."""
    from microscaled_precision_moe_gb300 import synth
    ids_n = ids.numpy()
    counts = np.bincount(ids_n.ravel(), minlength=shape.E)
    order = np.argsort(counts, kind="stable")
    picks = [int(e) for e in order[len(order) // 2:len(order) // 2 + n_experts]]
    items = []
    for e in picks:
        f = np.flatnonzero(ids_n.ravel() == e)
        tok = torch.from_numpy(f // shape.k)
        x = synth.moe_activations(shape, seed, rows=tok).float().numpy()
        w1, w2 = synth.moe_weights(shape, seed, experts=[e])
        items.append((e, x, w1.float().numpy()[0], w2.float().numpy()[0],
                      prob.numpy().ravel()[f]))
    return items


def _oracle_run(shape, items):
    """The oracle's NVFP4 expert path on the prepared sample: per-token
    quantisation of the routed rows, joint gate/up and W2 quantisation, fp64
    FC1, SwiGLU x prob, bf16, row amax, re-quantisation, fp64 FC2.
    Returns (algorithmic GEMM flops, seconds, description)."""
    from oracle import quant as Q
    from oracle import moe as MO
    from oracle import formats as F
    I, H = shape.I, shape.H
    flops, rows = 0, 0
    t0 = time.perf_counter()
    for e, x, w1, w2, p in items:
        qx, sx, tsx = Q.nvfp4_quantize_per_token(x)
        a = Q.nvfp4_dequantize(qx, sx, tsx)
        b1 = MO.dequant_weights_nvfp4(Q.nvfp4_quantize_joint([w1[None, :I], w1[None, I:]], 1))[0]
        b2 = MO.dequant_weights_nvfp4(Q.nvfp4_quantize_joint([w2[None]], 1))[0]
        with np.errstate(over="ignore"):
            d = MO.fc1_epilogue(a @ b1.T, p, I)
        amax = np.max(np.abs(d), axis=1).astype(np.float32)
        qd, sd, tsd = Q.nvfp4_quantize_per_token(d, amax)
        F.bf16_round(Q.nvfp4_dequantize(qd, sd, tsd) @ b2.T)
        n = x.shape[0]
        rows += n
        flops += 2 * n * H * 2 * I + 2 * n * I * H
    secs = time.perf_counter() - t0
    desc = (f"oracle NVFP4 expert path (numpy, fp64 GEMMs) over every routed row of "
            f"{len(items)} median-load expert(s): {rows} of {shape.T * shape.k} rows, "
            f"including their weight quantisation")
    return flops, secs, desc


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "nvfp4_fc1_fc2_dram_traffic.json")
GEMM_SOURCES = ("gemm2.cu", "gemm.cuh", "common.cuh")


def gemm_source_sha256() -> str:
    """Hash of the pair-GEMM sources the DRAM counters belong to: their code
    with comments and blank lines removed, so a change to a comment keeps the
    record while any change to the code drops it."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "microscaled_precision_moe_gb300", "csrc")
    code = []
    for f in GEMM_SOURCES:
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            line = line.split("//", 1)[0].rstrip()
            if line:
                code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()


def _gemm_traffic(path=TRAFFIC_FILE):
    """FC1 DRAM bytes per launch (read + write, ncu) of the headline workload
    from the committed counter record, if the GEMM sources are still the
    version those counters were taken on (else None)."""
    try:
        rec = json.load(open(path))
        if gemm_source_sha256() == rec["gemm_source_sha256"]:
            return int(rec["fc1_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        pass
    return None


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------- GPU helpers

def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _time_loop(fn, iters):
    s, e = _events(2)
    torch.cuda.synchronize()
    s.record()
    for _ in range(iters):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def _quantizer_lines(peak_hbm):
    """Quantiser throughput with rotating input buffers larger than L2."""
    from microscaled_precision_moe_gb300 import ops, synth
    out = {}
    # MXFP8 quantiser workload: 8288 x 2048 (row + column copies); 8 rotating
    # copies (8 x 34 MB) so each launch reads from HBM
    base = synth.mxfp8_quantizer_input(device="cuda")
    xs = [base.clone() for _ in range(8)]
    outs = [ops.mxfp8_quantize(x) for x in xs]
    M, K = base.shape
    byts = M * K * 2 + 2 * M * K + ops.scale_bytes(M, K // 32) + ops.scale_bytes(K, (M + 31) // 32)
    for i in range(3):
        ops.mxfp8_quantize(xs[i], out=outs[i])
    it = [0]

    def f():
        j = it[0] % 8
        ops.mxfp8_quantize(xs[j], out=outs[j])
        it[0] += 1
    ms_host = _time_loop(f, 80)
    # device time per launch: the eight launches captured once in a CUDA
    # graph and replayed, so the host's per-call cost does not pace the GPU
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for j in range(8):
            ops.mxfp8_quantize(xs[j], out=outs[j])
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            for j in range(8):
                ops.mxfp8_quantize(xs[j], out=outs[j])
    torch.cuda.synchronize()
    ms = _time_loop(g.replay, 10) / 8
    gbs = byts / (ms * 1e-3) / 1e9
    out["mxfp8_quantize_8288x2048_rowcol"] = {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2),
                                              "bytes": byts, "frac_hbm": round(gbs / peak_hbm, 3),
                                              "us_per_call_from_python": round(ms_host * 1e3, 2),
                                              "timing": "CUDA graph of 8 launches over 8 rotating "
                                                        "inputs (272 MB > L2), replayed"}
    del g
    # the same bytes moved by a plain device copy (torch's copy kernel), in
    # the same eight-launch graph: what a launch of this size reaches when it
    # does nothing but stream, i.e. the share of the gap that is the fixed
    # cost of a 15 us launch rather than the quantiser
    n_el = byts // 4                                      # bf16 in + bf16 out = 4 bytes per element
    srcs = [torch.empty(n_el, dtype=torch.bfloat16, device="cuda").fill_(1) for _ in range(8)]
    dsts = [torch.empty_like(t) for t in srcs]
    gc = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for j in range(8):
            dsts[j].copy_(srcs[j])
        torch.cuda.synchronize()
        with torch.cuda.graph(gc, stream=side):
            for j in range(8):
                dsts[j].copy_(srcs[j])
    torch.cuda.synchronize()
    ms_c = _time_loop(gc.replay, 10) / 8
    gbs_c = n_el * 4 / (ms_c * 1e-3) / 1e9
    out["mxfp8_quantize_8288x2048_rowcol"]["copy_same_bytes"] = {
        "us": round(ms_c * 1e3, 2), "GB/s": round(gbs_c, 1), "frac_hbm": round(gbs_c / peak_hbm, 3)}
    del gc, srcs, dsts
    del xs, outs
    # the same quantiser on a large input (65536 x 2048, 256 MB, the size of
    # an MXFP8 layer's permuted activations): streaming efficiency without the
    # fixed per-launch latency of the small case
    xl = synth.normal_bf16(0, synth.TID_X, (65536, 2048), "cuda")
    ol = ops.mxfp8_quantize(xl)
    for _ in range(3):
        ops.mxfp8_quantize(xl, out=ol)
    msl = _time_loop(lambda: ops.mxfp8_quantize(xl, out=ol), 20)
    Ml, Kl = xl.shape
    bl = Ml * Kl * 4 + ops.scale_bytes(Ml, Kl // 32) + ops.scale_bytes(Kl, (Ml + 31) // 32)
    gl = bl / (msl * 1e-3) / 1e9
    out["mxfp8_quantize_65536x2048_rowcol"] = {"GB/s": round(gl, 1), "us": round(msl * 1e3, 2),
                                               "bytes": bl, "frac_hbm": round(gl / peak_hbm, 3)}
    del xl, ol
    # NVFP4 per-token activation quantiser, 32768 x 7168 (470 MB > L2)
    x = synth.normal_bf16(0, synth.TID_X, (32768, 7168), "cuda")
    o = ops.nvfp4_quantize_per_token(x)
    for _ in range(3):
        ops.nvfp4_quantize_per_token(x, out=o)
    ms = _time_loop(lambda: ops.nvfp4_quantize_per_token(x, out=o), 30)
    byts = x.numel() * 2 + x.numel() // 2 + ops.scale_bytes(32768, 7168 // 16) + 32768 * 4
    gbs = byts / (ms * 1e-3) / 1e9
    out["nvfp4_quantize_per_token_32768x7168"] = {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2),
                                                  "bytes": byts, "frac_hbm": round(gbs / peak_hbm, 3)}
    del x, o
    torch.cuda.empty_cache()
    return out


def _single_expert_line(peak_fp4, peak_hbm, reps=3):
    """The single-expert NVFP4 case: 128 x 2048 activations (0.1 % of entries
    x50), 768 x 2048 gate and up weights quantised jointly, 128 x 1536 fp32
    output.  The per-token activation quantisation and the GEMM are timed
    separately.  Both fit in L2, so each launch reads one of a set of
    rotating copies whose total exceeds L2.  The launches are queued behind
    a spin kernel, so the events around them measure back-to-back device time
    instead of the host's per-call cost.  If the host took longer to queue
    them than the spin lasted, the line says so ("host_bound")."""
    from microscaled_precision_moe_gb300 import ops, synth
    from microscaled_precision_moe_gb300 import _lib as L
    x, wg, wu = synth.single_expert_inputs(device="cuda")
    M, K, N = x.shape[0], x.shape[1], 2 * wg.shape[0]
    n_q, n_g = 256, 96          # 256 x 0.67 MB and 96 x 2.6 MB of rotating data
    xs = [x.clone() for _ in range(n_q)]
    qs = [ops.nvfp4_quantize_per_token(xi) for xi in xs]
    qw, sw, tsw = ops.nvfp4_quantize_weight([wg[None].contiguous(), wu[None].contiguous()])
    ws = [(qw.clone(), sw.clone(), tsw.clone()) for _ in range(n_g)]
    outs = [torch.empty(M, N, dtype=torch.float32, device="cuda") for _ in range(n_g)]
    spin_cycles = int(4e7)      # about 20 ms at the SM clock

    def queued(fn, n):
        e0, s, e = _events(3)
        torch.cuda.synchronize()
        e0.record()
        torch.cuda._sleep(spin_cycles)
        s.record()
        t0 = time.perf_counter()
        for i in range(n):
            fn(i)
        host_ms = (time.perf_counter() - t0) * 1e3
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / n, host_ms > e0.elapsed_time(s)

    def quant(i):
        ops.nvfp4_quantize_per_token(xs[i], out=qs[i])

    def gemm(tile_m):
        def f(i):
            qx, sx, tsx = qs[i % n_q]
            q1, s1, t1 = ws[i]
            ops.moe_grouped_gemm(L.KIND_NVFP4, L.GROUP_M, L.EPI_F32, 1, M, N, K, None,
                                 qx, q1[0], sx, K // 16, s1, K // 16, outs[i],
                                 alpha_a=tsx, alpha_b=t1, tile_m=tile_m)
        return f

    out = {"workload": f"nvfp4_single_expert_M{M}_N{N}_K{K}",
           "timing": f"launches over rotating copies ({n_q} activation, {n_g} weight), queued "
                     "behind a spin kernel; median of the per-launch means of "
                     f"{reps} runs"}
    for i in range(3):
        quant(i)
    runs = [queued(quant, n_q) for _ in range(reps)]
    ms = float(np.median([r[0] for r in runs]))
    byts = M * K * 2 + M * K // 2 + ops.scale_bytes(M, K // 16) + M * 4
    out["quantize_per_token"] = {"us": round(ms * 1e3, 2), "bytes": byts,
                                 "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / peak_hbm, 3),
                                 "host_bound": any(r[1] for r in runs)}
    flops = 2 * M * N * K
    for tile_m, name in ((128, "gemm_one_cta"), (256, "gemm_cta_pair"), (L.TILE_SMALL_M, "gemm_small_m")):
        f = gemm(tile_m)
        for i in range(3):
            f(i)
        runs = [queued(f, n_g) for _ in range(reps)]
        ms = float(np.median([r[0] for r in runs]))
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 2), "flops": flops, "TFLOP/s": round(tf, 1),
                     "frac_fp4": round(tf / peak_fp4, 4), "host_bound": any(r[1] for r in runs)}
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0
    del xs, qs, ws, outs
    torch.cuda.empty_cache()
    return out


def _mxfp8_gemm_bounds(T, H, I, E, k, stage_ms, peak_fp8, peak_hbm):
    """Per GEMM of the MXFP8 step: algorithmic FLOPs (routed rows M = T k),
    the fewest HBM bytes it can move (each operand read once as stored, E4M3
    codes plus one E8M0 scale per 32, each output written once: bf16
    activations, fp32 weight gradients, and for FC1 the saved C = gate|up),
    the time each floor allows at the given peaks (TFLOP/s, GB/s), and the
    measured time's fraction of the larger floor."""
    M = T * k
    q = lambda n: n * (1 + 1 / 32)                       # MXFP8 operand bytes
    spec = {
        "fc1": (2 * M * 2 * I * H, q(M * H) + q(E * 2 * I * H) + 2 * M * I + 2 * M * 2 * I),
        "fc2": (2 * M * H * I, q(M * I) + q(E * H * I) + 2 * M * H),
        "fc2_dgrad": (2 * M * I * H, q(M * H) + q(E * I * H) + 2 * M * 2 * I + 2 * M * 2 * I),
        "fc2_wgrad": (2 * M * H * I, q(H * M) + q(I * M) + 4 * E * H * I),
        "fc1_dgrad": (2 * M * H * 2 * I, q(M * 2 * I) + q(H * E * 2 * I) + 2 * M * H),
        "fc1_wgrad": (2 * M * 2 * I * H, q(2 * I * M) + q(H * M) + 4 * E * 2 * I * H),
    }
    out, tot_ms, tot_floor = {}, 0.0, 0.0
    for name, (flops, byts) in spec.items():
        mma = flops / (peak_fp8 * 1e12) * 1e3
        hbm = byts / (peak_hbm * 1e9) * 1e3
        floor = max(mma, hbm)
        ms = stage_ms.get(name)
        out[name] = {"ms": ms, "flops": int(flops), "hbm_bytes": int(byts),
                     "mma_floor_ms": round(mma, 4), "hbm_floor_ms": round(hbm, 4),
                     "bound": "hbm" if hbm >= mma else "tensor",
                     "frac_of_bound": round(floor / ms, 3) if ms else None}
        if ms:
            tot_ms += ms
            tot_floor += floor
    out["all_gemms"] = {"ms": round(tot_ms, 4), "floor_ms": round(tot_floor, 4),
                        "frac_of_bound": round(tot_floor / tot_ms, 3) if tot_ms else None}
    return out


def _nvfp4_gemm_bounds(T, H, I, E, k, stage_ms, peak_fp4, peak_hbm):
    """FC1 and FC2 of the NVFP4 forward: algorithmic FLOPs over the routed
    rows M = T k, the fewest HBM bytes each can move (NVFP4 operands as
    stored: half a byte per element plus one E4M3 scale per 16; D and Y
    written once in bf16), each floor at the given peaks and the measured
    time's fraction of the larger floor."""
    M = T * k
    q = lambda n: n * (0.5 + 1 / 16)
    spec = {"fc1": (2 * M * 2 * I * H, q(M * H) + q(E * 2 * I * H) + 2 * M * I),
            "fc2": (2 * M * H * I, q(M * I) + q(E * H * I) + 2 * M * H)}
    out = {}
    for name, (flops, byts) in spec.items():
        mma = flops / (peak_fp4 * 1e12) * 1e3
        hbm = byts / (peak_hbm * 1e9) * 1e3
        ms = stage_ms.get(name)
        out[name] = {"ms": ms, "flops": int(flops), "hbm_bytes": int(byts),
                     "tensor_floor_ms": round(mma, 4), "hbm_floor_ms": round(hbm, 4),
                     "bound": "hbm" if hbm >= mma else "tensor",
                     "frac_of_bound": round(max(mma, hbm) / ms, 3) if ms else None}
    return out


def _mxfp8_layer_line(peak_fp8, steps=10, peak_hbm=None):
    from microscaled_precision_moe_gb300 import synth
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    s = synth.MOE_30B_BWD
    ids, prob = synth.routing(s)
    x = synth.moe_activations(s, device="cuda")
    w1, w2 = synth.moe_weights(s, device="cuda")
    dy = synth.moe_grad_out(s, device="cuda")
    L = MXFP8MoE(s.T, s.H, s.I, s.E, s.k)
    idc, prc = ids.cuda(), prob.cuda()

    def step(mark=None):
        if mark:
            mark(0)
        L.quantize_weights(w1, w2)
        L.forward(x, idc, prc, mark=mark)
        L.backward(dy, mark=mark)
    for _ in range(3):
        step()
    ms = _time_loop(step, steps)
    # per-stage times from a second, marked pass
    ns = len(MXFP8MoE.STEP_STAGES) + 1
    ev = [_events(ns) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        evi = ev[i]
        step(mark=lambda j, evi=evi: evi[j].record())
    torch.cuda.synchronize()
    stage = {n: round(float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)])), 4)
             for j, n in enumerate(MXFP8MoE.STEP_STAGES)}
    tf = L.gemm_flops() / (ms * 1e-3) / 1e12
    gemm_ms = sum(v for n, v in stage.items() if n.startswith("fc"))
    r = {"workload": s.name, "ms_per_step": round(ms, 3), "TFLOP/s": round(tf, 1),
         "frac_fp8_peak": round(tf / peak_fp8, 3),
         "gemm_TFLOP/s": round(L.gemm_flops() / (gemm_ms * 1e-3) / 1e12, 1),
         "stage_ms": stage,
         "gemm_bounds": (_mxfp8_gemm_bounds(s.T, s.H, s.I, s.E, s.k, stage, peak_fp8, peak_hbm)
                         if peak_hbm else None),
         "note": "whole fwd+bwd step (weight quantisation included) / GEMM algorithmic FLOPs"}
    del L, x, w1, w2, dy
    torch.cuda.empty_cache()
    return r


def _nvfp4_30b_line(peak_fp4, steps=10, peak_hbm=None):
    from microscaled_precision_moe_gb300 import synth
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    s = synth.MOE_30B
    ids, prob = synth.routing(s)
    x = synth.moe_activations(s, device="cuda")
    w1, w2 = synth.moe_weights(s, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    L = NVFP4MoE(s.T, s.H, s.I, s.E, s.k)
    idc, prc = ids.cuda(), prob.cuda()
    for _ in range(3):
        L.forward(x, idc, prc, W)
    ms = _time_loop(lambda: L.forward(x, idc, prc, W), steps)
    tf = sum(L.gemm_flops()) / (ms * 1e-3) / 1e12
    # per-stage times from a second, marked pass
    ns = len(NVFP4MoE.STAGES) + 1
    ev = [_events(ns) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        evi = ev[i]
        L.forward(x, idc, prc, W, mark=lambda j, evi=evi: evi[j].record())
    torch.cuda.synchronize()
    stage = {n: round(float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)])), 4)
             for j, n in enumerate(NVFP4MoE.STAGES)}
    r = {"workload": s.name, "ms_per_step": round(ms, 3), "TFLOP/s": round(tf, 1),
         "frac_fp4_peak": round(tf / peak_fp4, 3), "stage_ms": stage}
    if peak_hbm:
        r["gemm_bounds"] = _nvfp4_gemm_bounds(s.T, s.H, s.I, s.E, s.k, stage, peak_fp4, peak_hbm)
    del L, W, x, w1, w2
    torch.cuda.empty_cache()
    return r


def _nvfp4_online_line(peak_fp4, steps=10):
    """The headline layer with the single-pass FC2 of the miniTE report,
    section 5.6 (D quantised tile by tile against the running row amax, FC2
    weighing each tile by its outer scale), beside the two-pass layer the
    headline times; stage times from CUDA events."""
    from microscaled_precision_moe_gb300 import synth
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    s = synth.MOE_671B
    ids, prob = synth.routing(s)
    x = synth.moe_activations(s, device="cuda")
    w1, w2 = synth.moe_weights(s, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    del w1, w2
    torch.cuda.empty_cache()
    L = NVFP4MoE(s.T, s.H, s.I, s.E, s.k, fc2="online")
    idc, prc = ids.cuda(), prob.cuda()
    for _ in range(3):
        L.forward(x, idc, prc, W)
    nst = len(NVFP4MoE.STAGES) + 1
    ev = [_events(nst) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        evi = ev[i]
        L.forward(x, idc, prc, W, mark=lambda j, evi=evi: evi[j].record())
    torch.cuda.synchronize()
    tot = float(np.mean([ev[i][0].elapsed_time(ev[i][nst - 1]) for i in range(steps)]))
    st = {n: round(float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)])), 4)
          for j, n in enumerate(NVFP4MoE.STAGES)}
    fl1, fl2 = L.gemm_flops()
    r = {"workload": s.name + "_fc2_online", "ms_per_step": round(tot, 4),
         "TFLOP/s": round((fl1 + fl2) / (tot * 1e-3) / 1e12, 1),
         "fc2_TFLOP/s": round(fl2 / (st["fc2"] * 1e-3) / 1e12, 1),
         "fc2_frac_fp4": round(fl2 / (st["fc2"] * 1e-3) / 1e12 / peak_fp4, 3),
         "stage_ms": st,
         "note": "quant_d = the running-amax tile quantiser; fc2 = CTA pairs on 256 x 128 "
                 "tiles, each 256-column reduction tile weighed by its own outer scale"}
    del L, W, x
    torch.cuda.empty_cache()
    return r


def _bf16_bwd_gemm_bounds(T, H, I, E, k, stage_ms, peak_bf16, peak_hbm):
    """The four BF16 GEMMs of the backward, as `_mxfp8_gemm_bounds`: bf16
    operands read once (dY, D or dH, X, the transposed weights), C = gate|up
    read by the SwiGLU backward, dH and dX written in bf16, dW1 and dW2 in
    fp32; algorithmic FLOPs over the routed rows."""
    M = T * k
    spec = {
        "fc2_dgrad": (2 * M * I * H, 2 * M * H + 2 * E * H * I + 2 * M * 2 * I + 2 * M * 2 * I),
        "fc2_wgrad": (2 * M * H * I, 2 * M * H + 2 * M * I + 4 * E * H * I),
        "fc1_dgrad": (2 * M * 2 * I * H, 2 * M * 2 * I + 2 * E * 2 * I * H + 2 * M * H),
        "fc1_wgrad": (2 * M * 2 * I * H, 2 * M * 2 * I + 2 * M * H + 4 * E * 2 * I * H),
    }
    out, tot_ms, tot_floor = {}, 0.0, 0.0
    for name, (flops, byts) in spec.items():
        mma = flops / (peak_bf16 * 1e12) * 1e3
        hbm = byts / (peak_hbm * 1e9) * 1e3
        ms = stage_ms.get(name)
        out[name] = {"ms": ms, "flops": int(flops), "hbm_bytes": int(byts),
                     "tensor_floor_ms": round(mma, 4), "hbm_floor_ms": round(hbm, 4),
                     "bound": "hbm" if hbm >= mma else "tensor",
                     "frac_of_bound": round(max(mma, hbm) / ms, 3) if ms else None}
        if ms:
            tot_ms += ms
            tot_floor += max(mma, hbm)
    out["all_gemms"] = {"ms": round(tot_ms, 4), "floor_ms": round(tot_floor, 4),
                        "frac_of_bound": round(tot_floor / tot_ms, 3) if tot_ms else None}
    return out


def _nvfp4_bf16_bwd_line(peak_bf16, steps=10, peak_hbm=None):
    """BF16 backward of the NVFP4 layer (30B-shaped, 8192 tokens), both
    operand modes: the backward alone is timed (the forward that saves
    gate|up runs once before); the transposed weight copies are prepared once
    per weight update and timed separately."""
    from microscaled_precision_moe_gb300 import synth
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    s = synth.MOE_30B_BWD
    ids, prob = synth.routing(s)
    x = synth.moe_activations(s, device="cuda")
    w1, w2 = synth.moe_weights(s, device="cuda")
    dy = synth.moe_grad_out(s, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    L = NVFP4MoE(s.T, s.H, s.I, s.E, s.k)
    L.forward(x, ids.cuda(), prob.cuda(), W, save_for_backward=True)
    flops = L.backward_gemm_flops()
    r = {"workload": s.name, "note": "backward alone / algorithmic FLOPs of its four BF16 GEMMs"}
    for mode in NVFP4MoE.BACKWARD_MODES:
        prep = lambda: L.prepare_backward_weights(mode, w1=w1, w2=w2, w=W)
        for _ in range(2):
            prep()
        prep_ms = _time_loop(prep, 3)
        for _ in range(3):
            L.backward(dy, mode, x=x)
        nst = len(NVFP4MoE.BACKWARD_STAGES) + 1
        ev = [_events(nst) for _ in range(steps)]
        stream = torch.cuda.current_stream()
        st, en = _events(2)
        torch.cuda.synchronize()
        st.record(stream)
        for i in range(steps):
            evi = ev[i]
            L.backward(dy, mode, x=x, mark=lambda j, evi=evi: evi[j].record(stream))
        en.record(stream)
        torch.cuda.synchronize()
        ms = st.elapsed_time(en) / steps
        stage = {n: round(float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)])), 4)
                 for j, n in enumerate(NVFP4MoE.BACKWARD_STAGES)}
        tf = flops / (ms * 1e-3) / 1e12
        r[mode] = {"ms_per_step": round(ms, 3), "TFLOP/s": round(tf, 1),
                   "frac_bf16_peak": round(tf / peak_bf16, 3), "stage_ms": stage,
                   "prepare_weights_ms": round(prep_ms, 3),
                   "gpu_launches_per_step": NVFP4MoE.LAUNCHES_PER_BACKWARD[mode]}
        if peak_hbm:
            r[mode]["gemm_bounds"] = _bf16_bwd_gemm_bounds(s.T, s.H, s.I, s.E, s.k, stage,
                                                           peak_bf16, peak_hbm)
    del L, W
    torch.cuda.empty_cache()
    # the same modes after an MXFP8 forward
    from microscaled_precision_moe_gb300.moe import MXFP8MoE
    M8 = MXFP8MoE(s.T, s.H, s.I, s.E, s.k)
    M8.quantize_weights(w1, w2)
    M8.forward(x, ids.cuda(), prob.cuda())
    for mode in MXFP8MoE.BACKWARD_MODES:
        M8.prepare_backward_weights(mode, w1=w1, w2=w2)
        for _ in range(3):
            M8.backward_bf16(dy, mode)
        ms = _time_loop(lambda: M8.backward_bf16(dy, mode), steps)
        tf = flops / (ms * 1e-3) / 1e12
        r["mxfp8_fwd_" + mode] = {"ms_per_step": round(ms, 3), "TFLOP/s": round(tf, 1),
                                  "frac_bf16_peak": round(tf / peak_bf16, 3)}
    del M8, x, w1, w2, dy
    torch.cuda.empty_cache()
    return r


def _nvfp4_decode_line(peak_hbm, steps=20, experts=None, tokens=(64, 256)):
    """Decode / rollout-sized batches of the 671B-shaped layer (64 and 256
    tokens, Zipf load over 256 experts): the layer forward on the small-M
    kernel and, for comparison, on the CTA-pair kernel.  Bound: reading the
    active experts' FP4 weights (codes + E4M3 scales) once from HBM.
    experts: fewer experts (a small case for profiling)."""
    from microscaled_precision_moe_gb300 import synth, _lib as L
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights
    full = synth.MOE_671B if experts is None else synth.scaled(synth.MOE_671B, E=experts)
    w1, w2 = synth.moe_weights(full, device="cuda")
    W = NVFP4Weights.quantize(w1, w2)
    del w1, w2
    torch.cuda.empty_cache()
    r = {"workload": f"nvfp4_moe_fwd_decode_H7168_I2048_E{full.E}_k8_zipf1.1",
         "note": "layer forward; roofline = active experts' FP4 weight bytes / time vs measured HBM"}
    for T in tokens:
        s = synth.scaled(full, T=T)
        ids, prob = synth.routing(s)
        x = synth.moe_activations(s, device="cuda")
        idc, prc = ids.cuda(), prob.cuda()
        active = int(np.unique(ids.numpy()).size)
        wbytes = active * 3 * s.H * s.I * (0.5 + 1.0 / 16)
        for name, tm in (("small_m", L.TILE_SMALL_M), ("pair256", 256)):
            layer = NVFP4MoE(T, s.H, s.I, s.E, s.k, tile_m=tm)
            nst = len(NVFP4MoE.STAGES) + 1
            for _ in range(3):
                layer.forward(x, idc, prc, W)
            ev = [_events(nst) for _ in range(steps)]
            torch.cuda.synchronize()
            for i in range(steps):
                evi = ev[i]
                layer.forward(x, idc, prc, W, mark=lambda j, evi=evi: evi[j].record())
            torch.cuda.synchronize()
            tot = float(np.median([ev[i][0].elapsed_time(ev[i][nst - 1]) for i in range(steps)]))
            st = {n: round(float(np.median([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)])), 4)
                  for j, n in enumerate(NVFP4MoE.STAGES)}
            gemm_ms = st["fc1"] + st["fc2"]
            r[f"T{T}_{name}"] = {"active_experts": active, "ms": round(tot, 4),
                                 "gemm_ms": round(gemm_ms, 4),
                                 "weight_GB/s_in_gemms": round(wbytes / (gemm_ms * 1e-3) / 1e9, 1),
                                 "frac_hbm_gemms": round(wbytes / (gemm_ms * 1e-3) / 1e9 / peak_hbm, 3),
                                 "stage_ms": st}
            del layer
            torch.cuda.empty_cache()
    del W
    torch.cuda.empty_cache()
    return r


def _summary(line, peaks):
    """The secondary lines' key figures, compact, as the line's last key."""
    a = line.get("also", {})
    g = lambda d, *ks: _dig(d, ks)
    q = a.get("quantizers", {})
    sm = {"fc1_frac_fp4": line["roofline"]["frac"],
          "fc2_TFLOP/s": g(a, "stage_GBps_or_TFLOPs", "fc2_TFLOP/s"),
          "quant_frac_hbm": {k.split("_")[0] + "_" + k.split("_")[-2]: v.get("frac_hbm")
                             for k, v in q.items()},
          "mxfp8_step_ms": g(a, "mxfp8_layer_fwd_bwd", "ms_per_step"),
          "mxfp8_gemm_TFLOP/s": g(a, "mxfp8_layer_fwd_bwd", "gemm_TFLOP/s"),
          "mxfp8_gemm_frac_fp8_burst": None,
          "nvfp4_30b_ms": g(a, "nvfp4_layer_fwd_30b", "ms_per_step"),
          "nvfp4_30b_frac_fp4_burst": None,
          "fc2_online_ms": g(a, "nvfp4_layer_fwd_fc2_online", "stage_ms", "fc2"),
          "layer_fc2_online_ms": g(a, "nvfp4_layer_fwd_fc2_online", "ms_per_step"),
          "bf16_bwd_ms": {m: g(a, "nvfp4_layer_bf16_bwd", m, "ms_per_step")
                          for m in ("high_precision", "dequantized")},
          "decode_ms": {k: v.get("ms") for k, v in a.get("nvfp4_layer_decode", {}).items()
                        if isinstance(v, dict)},
          "single_expert_us": {k: v.get("us") for k, v in a.get("nvfp4_single_expert", {}).items()
                               if isinstance(v, dict)},
          "stage_frac_hbm": {k[:-9]: v for k, v in a.get("stage_GBps_or_TFLOPs", {}).items()
                             if k.endswith("_frac_hbm")}}
    fp8 = peaks["bf16"] * NOMINAL_FP8_OVER_BF16
    fp4 = peaks["bf16"] * NOMINAL_FP4_OVER_BF16
    if sm["mxfp8_gemm_TFLOP/s"]:
        sm["mxfp8_gemm_frac_fp8_burst"] = round(sm["mxfp8_gemm_TFLOP/s"] / fp8, 3)
    tf30 = g(a, "nvfp4_layer_fwd_30b", "TFLOP/s")
    if tf30:
        sm["nvfp4_30b_frac_fp4_burst"] = round(tf30 / fp4, 3)
    return sm


def _dig(d, ks):
    for k in ks:
        if not isinstance(d, dict) or k not in d:
            return None
        d = d[k]
    return d


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle sample")
    ap.add_argument("--case", choices=["headline", "slice", "mxfp8", "bf16bwd", "decode",
                                       "decode_slice", "quant", "single", "online"],
                    default="headline",
                    help="slice: 4096 tokens over 64 experts of the 671B shape (profiling); "
                         "mxfp8: the MXFP8 30B-shaped forward+backward step alone (profiling); "
                         "bf16bwd: the BF16 backward of the NVFP4 30B-shaped layer alone; "
                         "decode: 64 / 256-token batches of the 671B-shaped layer; "
                         "decode_slice: 64 tokens over 32 experts of that shape (profiling); "
                         "quant: the quantiser lines alone; "
                         "single: the single-expert 128 x 1536 x 2048 NVFP4 GEMM and its "
                         "activation quantisation; "
                         "online: the headline layer with the single-pass (online amax) FC2")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from microscaled_precision_moe_gb300 import synth
    shape = synth.MOE_671B
    if args.case == "slice":
        shape = synth.scaled(shape, T=4096, E=64, name="nvfp4_moe_fwd_T4096_H7168_I2048_E64_k8_zipf1.1")
    peaks = _peaks()
    peak_fp4 = peaks["bf16"] * NOMINAL_FP4_OVER_BF16
    peak_fp4_sus = peaks["bf16_sus"] * NOMINAL_FP4_OVER_BF16
    peak_fp8_sus = peaks["bf16_sus"] * NOMINAL_FP8_OVER_BF16
    cfg = {"workload": shape.name, "tokens": shape.T, "hidden": shape.H,
           "intermediate": shape.I, "experts": shape.E, "top_k": shape.k,
           "expert_load": "Zipf(1.1) via Gumbel-top-k", "weights": "N(0,0.01), 1e-4 outliers x100",
           "l2": "no flush: inputs exceed L2 (activations %d MB, FP4 weights %.1f GB)" % (
               shape.T * shape.H * 2 // 2 ** 20, shape.E * 3 * shape.H * shape.I * 0.5625 / 1e9)}

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        ids, prob = synth.routing(shape)
        items = _oracle_prepare(shape, ids, prob, n_experts=1)
        for _ in range(args.warmup):                  # the W untimed steps the line reports
            _oracle_run(shape, items)
        vals, descs = [], []
        t_all = time.perf_counter()
        for _ in range(args.steps):
            fl, sec, desc = _oracle_run(shape, items)
            vals.append(fl / sec / 1e12)
            descs.append(desc)
        wall = time.perf_counter() - t_all
        v = float(np.median(vals))
        line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(wall / args.steps * 1e3, 1), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg,
                "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": _cores(),
                                 "kind": "oracle", "sample": descs[0]},
                "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    dist, rank, world = _dist()
    dev = torch.cuda.current_device()
    from microscaled_precision_moe_gb300 import build
    build.build()
    if args.case == "mxfp8":
        r = _mxfp8_layer_line(peak_fp8_sus, steps=args.steps, peak_hbm=peaks["hbm"])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["TFLOP/s"], "unit": "TFLOP/s",
                              "n_gpus": world, "steps": args.steps, "warmup": 3,
                              "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                              "dtype": "mxfp8", "config": {"workload": r["workload"]},
                              "note": r["note"], "gemm_TFLOP/s": r["gemm_TFLOP/s"],
                              "stage_ms": r["stage_ms"], "gemm_bounds": r["gemm_bounds"]}),
                  flush=True)
        return 0
    if args.case == "quant":
        r = _quantizer_lines(peaks["hbm"])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["mxfp8_quantize_8288x2048_rowcol"]["GB/s"],
                              "unit": "GB/s", "n_gpus": world, "higher_is_better": True,
                              "dtype": "mxfp8", "config": {"workload": "mxfp8_quantize_8288x2048_rowcol"},
                              "quantizers": r}), flush=True)
        return 0
    if args.case == "online":
        r = _nvfp4_online_line(peaks["bf16"] * NOMINAL_FP4_OVER_BF16, steps=args.steps)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["TFLOP/s"], "unit": "TFLOP/s",
                              "n_gpus": world, "steps": args.steps, "warmup": 3,
                              "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                              "dtype": "nvfp4", "config": {"workload": r["workload"]},
                              "online": r}), flush=True)
        return 0
    if args.case == "single":
        r = _single_expert_line(peak_fp4_sus, peaks["hbm"])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["gemm_one_cta"]["us"], "unit": "us",
                              "n_gpus": world, "higher_is_better": False, "dtype": "nvfp4",
                              "config": {"workload": r["workload"]}, "single_expert": r}),
                  flush=True)
        return 0
    if args.case in ("decode", "decode_slice"):
        r = (_nvfp4_decode_line(peaks["hbm"], steps=args.steps) if args.case == "decode" else
             _nvfp4_decode_line(peaks["hbm"], steps=args.steps, experts=32, tokens=(64,)))
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["T64_small_m"]["ms"], "unit": "ms",
                              "n_gpus": world, "steps": args.steps, "warmup": 3,
                              "higher_is_better": False, "dtype": "nvfp4",
                              "config": {"workload": r["workload"]}, "decode": r}), flush=True)
        return 0
    if args.case == "bf16bwd":
        r = _nvfp4_bf16_bwd_line(peaks["bf16_sus"], steps=args.steps, peak_hbm=peaks["hbm"])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["dequantized"]["TFLOP/s"],
                              "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                              "warmup": 3, "ms_per_step": r["dequantized"]["ms_per_step"],
                              "higher_is_better": True, "dtype": "bf16",
                              "config": {"workload": r["workload"]}, "modes": r}), flush=True)
        return 0
    from microscaled_precision_moe_gb300 import ops
    from microscaled_precision_moe_gb300.moe import NVFP4MoE, NVFP4Weights

    # ---- inputs (seeded, synthetic) and weights quantised once
    ids, prob = synth.routing(shape)
    x = synth.moe_activations(shape, device="cuda")
    w1, w2 = synth.moe_weights(shape, device="cuda")
    torch.cuda.synchronize()
    W = NVFP4Weights.quantize(w1, w2)
    for _ in range(2):
        NVFP4Weights.quantize(w1, w2)
    t_wq = _time_loop(lambda: NVFP4Weights.quantize(w1, w2), 3)
    wbytes = (w1.numel() + w2.numel()) * 2.5 + (w1.numel() + w2.numel()) // 16
    del w1, w2
    torch.cuda.empty_cache()
    idc, prc = ids.cuda(), prob.cuda()
    layer = NVFP4MoE(shape.T, shape.H, shape.I, shape.E, shape.k)
    fl1, fl2 = layer.gemm_flops()
    flops = fl1 + fl2

    for _ in range(args.warmup):
        layer.forward(x, idc, prc, W)
    torch.cuda.synchronize()
    assert ops.get_device_status() == 0

    # ---- timed region: K steps, per-stage events on the launching stream
    nst = len(NVFP4MoE.STAGES) + 1
    ev = [_events(nst) for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    start, end = _events(2)
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        start.record(stream)
        for i in range(args.steps):
            evi = ev[i]
            layer.forward(x, idc, prc, W, mark=lambda j, evi=evi: evi[j].record(stream))
        end.record(stream)
        torch.cuda.synchronize()
        _barrier(dist)
    ms = start.elapsed_time(end) / args.steps
    ms = _max_over_ranks(dist, ms)
    stage_ms = {name: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)]))
                for j, name in enumerate(NVFP4MoE.STAGES)}
    value = world * flops / (ms * 1e-3) / 1e12
    # algorithmic bytes of the HBM-bound stages, for their GB/s (R routed
    # rows, r_pad rows after per-expert padding; one NVFP4 row of n elements
    # is n/2 code bytes, n/16 scale bytes and a 4-byte token scale)
    R = shape.T * shape.k
    r_pad = int(layer.seg[0][shape.E].item())
    nv_row = lambda n: n // 2 + n // 16 + 4
    stage_bytes = {
        "quant_x": shape.T * shape.H * 2 + r_pad * (nv_row(shape.H) + 4) + r_pad * 4 + R * 4,
        "quant_d": r_pad * (shape.I * 2 + 4) + r_pad * nv_row(shape.I),
        "combine": R * shape.H * 2 + R * 4 + shape.T * shape.H * 2}

    # ---- e2e through the public API: every step uploads its inputs from
    # pinned host memory and downloads its output; double-buffered, so step
    # i+1's upload and step i-1's download run on two copy streams (one per
    # direction, so both directions move at once) while step i computes (a
    # serving loop's schedule)
    xh = x.cpu().pin_memory()
    idh, prh = ids.pin_memory(), prob.pin_memory()
    outh = [torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    idd = [torch.empty_like(idc) for _ in range(2)]
    prd = [torch.empty_like(prc) for _ in range(2)]
    od = [torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device=x.device) for _ in range(2)]
    cs = torch.cuda.current_stream()
    xs, ys = torch.cuda.Stream(), torch.cuda.Stream()     # uploads, downloads

    # the output leaves in E2E_CHUNKS token ranges, each copied to the host
    # as soon as the layer has combined it (forward's on_chunk), so only the
    # last range's copy follows the last step's compute
    E2E_CHUNKS = 8
    chunk_ev = [[torch.cuda.Event() for _ in range(E2E_CHUNKS)] for _ in range(2)]

    def e2e_run(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def upload(b):
            with torch.cuda.stream(xs):
                xs.wait_event(comp_done[b])            # the step that read these buffers is done
                xd[b].copy_(xh, non_blocking=True)
                idd[b].copy_(idh, non_blocking=True)
                prd[b].copy_(prh, non_blocking=True)
                in_ready[b].record(xs)
        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload((i + 1) % 2)
            cs.wait_event(in_ready[b])
            cs.wait_event(out_done[b])                 # od[b]'s previous download is done
            def on_chunk(j, t0, t1, b=b):
                chunk_ev[b][j].record(cs)
                with torch.cuda.stream(ys):
                    ys.wait_event(chunk_ev[b][j])
                    outh[b][t0:t1].copy_(od[b][t0:t1], non_blocking=True)
            layer.forward(xd[b], idd[b], prd[b], W, out=od[b], out_chunks=E2E_CHUNKS,
                          on_chunk=on_chunk)
            comp_done[b].record(cs)
            with torch.cuda.stream(ys):
                out_done[b].record(ys)
        cs.wait_stream(xs)
        cs.wait_stream(ys)
    e2e_run(3)
    n_e2e = max(4, args.steps)
    torch.cuda.synchronize()
    t_e2e = time.perf_counter()
    s0, s1 = _events(2)
    s0.record(cs)
    e2e_run(n_e2e)
    s1.record(cs)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / n_e2e
    e2e_wall_ms = (time.perf_counter() - t_e2e) * 1e3 / n_e2e
    h2d = xh.numel() * 2 + idh.numel() * 4 + prh.numel() * 4
    d2h = outh[0].numel() * 2

    # ---- roofline of the dominant kernel (FC1 grouped GEMM, tensor bound)
    fc1_ms = stage_ms["fc1"]
    ach = fl1 / (fc1_ms * 1e-3) / 1e12
    traffic = _gemm_traffic() if args.case == "headline" else None
    # burst peak: the timed region lasts a fraction of a second at the
    # maximum SM clock (the clock record says so), not a seconds-long loop
    # under the power cap
    roof = {"bound": "tensor", "kernel": "grouped_gemm_pair_kernel<NVFP4, SWIGLU> (FC1)",
            "achieved": round(ach, 1), "peak": round(peak_fp4, 1), "unit": "TFLOP/s",
            "frac": round(ach / peak_fp4, 4), "traffic": traffic,
            "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
            "peak_source": f"{peaks['src']} burst bf16 x {NOMINAL_FP4_OVER_BF16:g} "
                           f"(dense FP4/BF16 nominal ratio)",
            "frac_of_sustained_peak": round(ach / peak_fp4_sus, 4),
            "per_launch_flops": fl1}

    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4", "data": "synthetic (seeded counter-based generator)",
            "config": cfg, "parallelism": "replicas" if world > 1 else "single",
            "clocks": clk.summary(), "roofline": roof,
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "gemm_bounds": _nvfp4_gemm_bounds(shape.T, shape.H, shape.I, shape.E, shape.k,
                                              stage_ms, peak_fp4, peaks["hbm"]),
            "gpu_launches": NVFP4MoE.LAUNCHES_PER_FORWARD * args.steps,
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 4), "host_wall_ms_per_step": round(e2e_wall_ms, 4),
                    "steps": n_e2e,
                    "schedule": "pinned uploads and downloads on one copy stream each, double-buffered "
                                "against the compute stream; the output is combined in "
                                f"{E2E_CHUNKS} token ranges and each range is downloaded as soon as "
                                "it is combined"},
            "weight_quantize": {"ms": round(t_wq, 3),
                                "GB/s": round(wbytes / (t_wq * 1e-3) / 1e9, 1)}}
    del xh, outh, xd, od, layer, W, x
    torch.cuda.empty_cache()

    if rank == 0 and not args.no_cpu:
        fl_s, sec_s, desc = _oracle_run(shape, _oracle_prepare(shape, ids, prob, n_experts=3))
        line["cpu_baseline"] = {"value": round(fl_s / sec_s / 1e12, 6), "unit": "TFLOP/s",
                                "cores": _cores(), "kind": "oracle", "sample": desc}
    if not args.no_also:
        also = {"quantizers": _quantizer_lines(peaks["hbm"])}
        also["mxfp8_layer_fwd_bwd"] = _mxfp8_layer_line(peak_fp8_sus, peak_hbm=peaks["hbm"])
        also["nvfp4_layer_fwd_30b"] = _nvfp4_30b_line(peak_fp4_sus, peak_hbm=peaks["hbm"])
        also["nvfp4_layer_fwd_fc2_online"] = _nvfp4_online_line(peak_fp4)
        also["nvfp4_layer_bf16_bwd"] = _nvfp4_bf16_bwd_line(peaks["bf16_sus"], peak_hbm=peaks["hbm"])
        also["nvfp4_layer_decode"] = _nvfp4_decode_line(peaks["hbm"])
        try:
            also["nvfp4_single_expert"] = _single_expert_line(peak_fp4_sus, peaks["hbm"])
        except Exception as exc:       # a secondary line never costs the main one
            also["nvfp4_single_expert"] = {"error": f"{type(exc).__name__}: {exc}"}
        also["stage_GBps_or_TFLOPs"] = {
            "fc1_TFLOP/s": round(ach, 1),
            "fc2_TFLOP/s": round(fl2 / (stage_ms["fc2"] * 1e-3) / 1e12, 1)}
        for name, nb in stage_bytes.items():
            gbs = nb / (stage_ms[name] * 1e-3) / 1e9
            also["stage_GBps_or_TFLOPs"][f"{name}_GB/s"] = round(gbs, 1)
            also["stage_GBps_or_TFLOPs"][f"{name}_frac_hbm"] = round(gbs / peaks["hbm"], 3)
        also["stage_GBps_or_TFLOPs"]["bytes"] = {
            **stage_bytes, "rows": R, "padded_rows": r_pad,
            "counted": "quant_x: the bf16 tokens read once, every padded row written "
                       "(NVFP4 codes, scales, token scale, zeroed amax slot), the row and slot "
                       "maps read; "
                       "quant_d: bf16 D and the amax read, NVFP4 D written (padded rows); "
                       "combine: the routed rows of Y and the inverse map read, the output "
                       "written"}
        line["also"] = also
        line["summary"] = _summary(line, peaks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
