"""Host-side logic of bench.py that decides what a bench line reports: the peaks it divides
by, which committed DRAM-traffic records still apply, and the clock summary that marks a run
as throttled.  CPU only: no GPU, no nvidia-smi."""
import hashlib
import json
import os

import bench


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6486.5, "bf16_tflops": 1805.2, "bf16_tflops_sustained": 1405.8, "x": 1}))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert peaks == {"hbm_gbs": 6486.5, "bf16_tflops": 1805.2, "bf16_tflops_sustained": 1405.8}


def test_traffic_record_applies_only_while_its_source_is_unchanged(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# comment\n"
        f"fused_fwd_gemm k.cu {sha} 53564160 config2\n"
        f"decode_gemv k.cu {'0' * 64} 126204672 config4\n")
    assert bench.traffic_records() == {("fused_fwd_gemm", "config2"): 53564160.0}
    src.write_text("kernel v2\n")
    assert bench.traffic_records() == {}


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _clock_summary(tmp_path, lines):
    c = bench.Clocks(0)
    c.path = str(tmp_path / "clocks.csv")
    (tmp_path / "clocks.csv").write_text("".join(l + "\n" for l in lines))
    c.f = open(str(tmp_path / "sink"), "w")
    c.proc = _FakeProc()
    return c.stop()


def test_clock_summary_median_max_and_reasons(tmp_path):
    na = "Not Active"
    lines = [f"0, {mhz}, 2032, 900.5, 0x0, {na}, {na}, {na}, {cap}"
             for mhz, cap in ((2032, na), (1965, "Active"), (2032, na))]
    lines.insert(1, "garbage line")
    s = _clock_summary(tmp_path, lines)
    assert s == {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    hot = [f"0, 1500, 2032, 1000, 0x48, {na}, Active, {na}, {na}"]
    assert _clock_summary(tmp_path, hot)["reasons"] == ["hw_thermal_slowdown"]
    assert _clock_summary(tmp_path, []) is None
