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


def test_clock_summary_without_samples():
    s = _summary([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["unsampled"]


def test_gemm_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed counters only while the GEMM
    sources hash to the value recorded with them; an edited source or a
    missing summary gives None."""
    import hashlib
    csrc = tmp_path / "microscaled_precision_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, body in (("gemm2.cu", b"pair"), ("gemm.cuh", b"decl"), ("common.cuh", b"util")):
        (csrc / name).write_bytes(body)
    digest = hashlib.sha256(b"pair" + b"decl" + b"util").hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "nvfp4_fc1_fc2_T32768_H7168_I2048_E256_dram_traffic.md").write_text(
        f"# counters\n\nfc1_traffic_bytes_per_launch: 123456\ngemm_source_sha256: {digest}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._gemm_traffic() == 123456
    (csrc / "gemm2.cu").write_bytes(b"pair, edited")
    assert bench._gemm_traffic() is None
    (prof / "nvfp4_fc1_fc2_T32768_H7168_I2048_E256_dram_traffic.md").unlink()
    assert bench._gemm_traffic() is None


def test_gemm_traffic_of_the_committed_tree_is_consistent():
    """In this tree the recorded hash predates the current pair kernel, so the
    bench must report no traffic; if the counters are recaptured and the hash
    updated, the value read back is the recorded one."""
    import hashlib
    csrc = os.path.join(ROOT, "microscaled_precision_moe_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, f), "rb").read()
                   for f in ("gemm2.cu", "gemm.cuh", "common.cuh"))
    text = open(os.path.join(ROOT, "profiles",
                             "nvfp4_fc1_fc2_T32768_H7168_I2048_E256_dram_traffic.md")).read()
    recorded = [l.split(": ", 1)[1].strip() for l in text.split("\n")
                if l.startswith("gemm_source_sha256: ")]
    assert len(recorded) == 1
    t = bench._gemm_traffic()
    if hashlib.sha256(src).hexdigest() == recorded[0]:
        assert isinstance(t, int) and t > 0
    else:
        assert t is None
