"""Host logic of bench.py that needs no GPU: the clock-record summary that
decides whether a timed run saw a throttle reason (CPU only)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(lines):
    c = bench.ClockSampler(0)
    c.lines = list(lines)
    return c.summary()


def test_clock_summary_median_max_and_power_cap():
    rows = ["0, 2032, 2070, 1100.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 2040, 2070, 1180.25, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 1995, 2070, 1390.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    s = _summary(rows)
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_clock_summary_reports_rejecting_reasons_and_skips_bad_lines():
    rows = ["0, 1500, 2070, 900.0, 0x08, Active, Not Active, Not Active, Not Active",
            "0, 1400, 2070, 900.0, 0x40, Not Active, Active, Active, Not Active",
            "garbage",
            "0, [N/A], 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            ""]
    s = _summary(rows)
    assert s["samples"] == 2 and s["sm_mhz"] == 1450.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_keeps_the_samples_of_the_timed_region():
    """Samples that arrived before the timed region started (the idle clock
    while nvidia-smi came up) are left out; with none after, all count."""
    idle = "0, 345, 2070, 120.0, 0x01, Not Active, Not Active, Not Active, Not Active"
    busy = "0, 2070, 2070, 1100.0, 0x00, Not Active, Not Active, Not Active, Not Active"
    c = bench.ClockSampler(0)
    c.lines = [idle, busy, busy]
    c.first = 1
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2070.0
    c.lines, c.first = [idle], 1
    assert c.summary()["samples"] == 1


def test_clock_summary_without_samples():
    s = _summary([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["unsampled"]


def test_gemm_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed counter record (a JSON data
    file, not the markdown report) only while the GEMM sources' code hashes to
    the value recorded with it: an edited comment keeps the record, edited
    code, a malformed or a missing record gives None."""
    import hashlib
    import json
    csrc = tmp_path / "microscaled_precision_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, body in (("gemm2.cu", "pair();  // the pair kernel\n\n"),
                       ("gemm.cuh", "/* declarations\n   of the args */\ndecl;\n"),
                       ("common.cuh", "util();\n")):
        (csrc / name).write_text(body)
    digest = hashlib.sha256(b"pair();\ndecl;\nutil();").hexdigest()
    rec = tmp_path / "traffic.json"
    rec.write_text(json.dumps({"fc1_bytes_per_launch": 123456, "gemm_source_sha256": digest}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.gemm_source_sha256() == digest
    assert bench._gemm_traffic(str(rec)) == 123456
    (csrc / "gemm2.cu").write_text("pair();  // the CTA-pair kernel, reworded\n")
    assert bench._gemm_traffic(str(rec)) == 123456
    rec.write_text("{not json")
    assert bench._gemm_traffic(str(rec)) is None
    rec.write_text(json.dumps({"fc1_bytes_per_launch": 123456, "gemm_source_sha256": digest}))
    (csrc / "gemm2.cu").write_text("pair(1);\n")
    assert bench._gemm_traffic(str(rec)) is None
    rec.unlink()
    assert bench._gemm_traffic(str(rec)) is None


def test_gemm_traffic_of_the_committed_tree_is_consistent():
    """The bench reports the recorded FC1 traffic exactly when the committed
    record's hash is the current sources' hash, and nothing otherwise."""
    import json
    t = bench._gemm_traffic()
    if not os.path.exists(bench.TRAFFIC_FILE):
        assert t is None
        return
    rec = json.load(open(bench.TRAFFIC_FILE))
    if rec["gemm_source_sha256"] == bench.gemm_source_sha256():
        assert t == int(rec["fc1_bytes_per_launch"]) and t > 0
    else:
        assert t is None


def test_summary_of_a_line():
    """The compact summary (the line's last key) reads the secondary lines
    and tolerates missing ones."""
    peaks = {"bf16": 1900.0, "bf16_sus": 1700.0, "hbm": 6800.0}
    line = {"roofline": {"frac": 0.5},
            "also": {"quantizers": {"mxfp8_quantize_8288x2048_rowcol": {"frac_hbm": 0.6}},
                     "mxfp8_layer_fwd_bwd": {"ms_per_step": 2.5, "gemm_TFLOP/s": 1900.0},
                     "stage_GBps_or_TFLOPs": {"fc2_TFLOP/s": 5000.0, "quant_x_frac_hbm": 0.95}}}
    s = bench._summary(line, peaks)
    assert s["fc1_frac_fp4"] == 0.5 and s["fc2_TFLOP/s"] == 5000.0
    assert s["mxfp8_gemm_frac_fp8_burst"] == 0.5
    assert s["stage_frac_hbm"] == {"quant_x": 0.95}
    assert s["nvfp4_30b_ms"] is None and s["nvfp4_30b_frac_fp4_burst"] is None
    assert bench._summary({"roofline": {"frac": 0.1}}, peaks)["decode_ms"] == {}


def test_mxfp8_gemm_bounds_bytes_and_floors():
    """Hand-counted case: 32 tokens, top-2 (64 routed rows), H 64, I 32,
    2 experts.  MXFP8 operand = 1 byte per element plus 1/32 byte of scale."""
    import bench
    st = {"fc1": 1e-3, "fc2": 1e-3, "fc2_dgrad": 1e-3, "fc2_wgrad": 1e-3, "fc1_dgrad": 1e-3,
          "fc1_wgrad": 2e-3}
    r = bench._mxfp8_gemm_bounds(32, 64, 32, 2, 2, st, peak_fp8=1.0, peak_hbm=1.0)
    # fc2 wgrad: dY column copy 64 x 64, D column copy 32 x 64, dW2 fp32 2 x 64 x 32
    assert r["fc2_wgrad"]["hbm_bytes"] == 4224 + 2112 + 16384
    assert r["fc2_wgrad"]["flops"] == 2 * 64 * 64 * 32
    # fc1: X 64 x 64, W1 2 x 64 x 64 (codes + scales), D 64 x 32 bf16, C 64 x 64 bf16
    assert r["fc1"]["hbm_bytes"] == 4224 + 8448 + 4096 + 8192
    # 1 TFLOP/s and 1 GB/s: the floors in ms are flops / 1e9 and bytes / 1e6
    assert r["fc1"]["mma_floor_ms"] == round(2 * 64 * 64 * 64 / 1e9, 4)
    assert r["fc1"]["hbm_floor_ms"] == round(24960 / 1e6, 4)
    assert r["fc1"]["bound"] == "hbm"
    # fc1 wgrad: dH and X column copies 64 x 64 each, dW1 fp32 2 x 64 x 64
    assert r["fc1_wgrad"]["hbm_bytes"] == 4224 + 4224 + 32768
    assert r["fc1_wgrad"]["frac_of_bound"] == round(41216 / 1e6 / 2e-3, 3)
    tot = sum(st.values())
    assert abs(r["all_gemms"]["ms"] - tot) < 1e-9


def test_nvfp4_gemm_bounds_headline_shape():
    """The headline layer's FC2 writes Y in bf16 and reads every expert's
    FP4 W2: at the measured peaks its HBM floor exceeds its FP4 floor, while
    FC1 stays bound by the tensor cores."""
    import bench
    r = bench._nvfp4_gemm_bounds(32768, 7168, 2048, 256, 8, {"fc1": 2.8, "fc2": 1.7},
                                 peak_fp4=11373.0, peak_hbm=6790.0)
    M = 32768 * 8
    assert r["fc2"]["hbm_bytes"] == int(M * 2048 * 0.5625 + 256 * 7168 * 2048 * 0.5625
                                        + 2 * M * 7168)
    assert r["fc1"]["bound"] == "tensor" and r["fc2"]["bound"] == "hbm"
    assert 0.4 < r["fc2"]["frac_of_bound"] < 0.7


def test_bf16_backward_gemm_bounds_bytes():
    """Hand-counted case: 64 routed rows, H 64, I 32, 2 experts, bf16
    operands and outputs, fp32 weight gradients."""
    import bench
    st = {"fc2_dgrad": 1e-3, "fc2_wgrad": 1e-3, "fc1_dgrad": 1e-3, "fc1_wgrad": 1e-3}
    r = bench._bf16_bwd_gemm_bounds(32, 64, 32, 2, 2, st, peak_bf16=1.0, peak_hbm=1.0)
    # FC2 dgrad: dY 64 x 64, W2 2 x 64 x 32, C 64 x 64 read, dH 64 x 64 written (bf16)
    assert r["fc2_dgrad"]["hbm_bytes"] == 8192 + 8192 + 8192 + 8192
    # FC1 wgrad: dH 64 x 64 and X 64 x 64 (bf16), dW1 2 x 64 x 64 fp32
    assert r["fc1_wgrad"]["hbm_bytes"] == 8192 + 8192 + 32768
    assert r["fc1_dgrad"]["flops"] == 2 * 64 * 64 * 64
    assert abs(r["all_gemms"]["ms"] - 4e-3) < 1e-12
