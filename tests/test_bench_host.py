"""Host logic of bench.py that needs no GPU: the DRAM-traffic record is used
only while the kernel sources it was measured on are unchanged, the clock
sampler's parsing of nvidia-smi lines (median SM clock, throttle reasons), the
roofline denominators (measured peaks, else the stated fallback) and the timing
statistics."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _write_record(root, sources, kernels):
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "gemm_traffic.json"), "w") as fh:
        json.dump({"sources": sources, "sources_sha256": h.hexdigest(), "kernels": kernels}, fh)


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k") == (None, None)          # no record
    os.makedirs(tmp_path / "src")
    (tmp_path / "src" / "a.cu").write_text("kernel a")
    (tmp_path / "src" / "b.cuh").write_text("header b")
    _write_record(str(tmp_path), ["src/a.cu", "src/b.cuh"],
                  {"k": {"dram_bytes_per_launch": 1234, "workload": [1, 2, 3]}})
    assert bench.recorded_traffic("k") == (1234, [1, 2, 3])
    assert bench.recorded_traffic("other") == (None, None)       # kernel not in the record
    (tmp_path / "src" / "b.cuh").write_text("header b, changed")
    assert bench.recorded_traffic("k") == (None, None)           # counters are stale


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


class _Thread:
    def join(self, timeout=None):
        pass


def _sampler(lines):
    s = bench.ClockSampler(None)
    s.proc, s.thread, s.lines = _Proc(), _Thread(), lines
    return s.stop()


def test_clock_sampler_parses_clocks_and_reasons():
    na = "Not Active"
    lines = [
        f"2070, 2070, 1100.5, {na}, {na}, {na}, {na}",
        f"1965, 2070, 1398.0, {na}, {na}, {na}, Active",
        f"2040, 2070, 1350.2, {na}, {na}, {na}, {na}",
        "garbage line",
        f"[N/A], 2070, 1.0, {na}, {na}, {na}, {na}",
    ]
    c = _sampler(lines)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2040.0
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    c = _sampler([f"1500, 2070, 900, Active, {na}, Active, {na}"])
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler([]) is None


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(None)
    assert s.stop() is None                                        # never started


def test_peaks_measured_else_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6796.2, "bf16_tflops": 1855.4, "bf16_tflops_sustained": 1700.0}))
    p = bench.peaks()
    assert p == {"hbm_gbs": 6796.2, "bf16": 1855.4, "bf16_sus": 1700.0, "source": "measured"}


def test_timing_statistics():
    """Median, p10/p90 and the mean of the middle 80 % of a set of repetitions:
    readings that sit on two event steps (2.048 us apart) in a 60/40 split have
    their median on the lower step and the trimmed mean between the two."""
    ts = [0.006144] * 60 + [0.008192] * 40
    st = bench.stats_us(ts)
    assert st["n"] == 100
    assert st["us"] == 6.14 and st["p10"] == 6.14 and st["p90"] == 8.19
    # the middle 80 repetitions: 50 on the lower step, 30 on the upper one
    assert abs(st["mean_mid80"] - (50 * 6.144 + 30 * 8.192) / 80) < 0.01
    one = bench.stats_us([1.0])
    assert one["us"] == one["mean_mid80"] == 1000.0
