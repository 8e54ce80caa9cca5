"""Host logic of bench.py that decides what its JSON line reports, on the CPU: the kernel-source
hash that keeps a recorded DRAM-traffic figure valid only for the code it was measured on, the
reading of that figure, the clock-sample summary (median SM clock, throttle reasons inside the
timed region) and the fallback peaks."""
import os
import shutil

import pytest

import bench


@pytest.fixture
def src_copy(tmp_path, monkeypatch):
    """bench.ROOT pointed at a copy of the kernel sources."""
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(path, fn):
    txt = path.read_text(encoding="utf-8")
    path.write_text(fn(txt), encoding="utf-8")


def test_kernel_hash_ignores_comments_and_blank_space(src_copy):
    h0 = bench.kernel_hash()
    first = src_copy / bench.KERNEL_SOURCES[0]
    _edit(first, lambda t: "// a new comment line\n" + t.replace("\n", "\n\n", 3) + "\n/* block comment */\n")
    assert bench.kernel_hash() == h0


def test_kernel_hash_changes_with_the_code(src_copy):
    h0 = bench.kernel_hash()
    last = src_copy / bench.KERNEL_SOURCES[-1]
    _edit(last, lambda t: t + "\nnamespace coda { constexpr int kHashProbe = 1; }\n")
    assert bench.kernel_hash() != h0


def test_recorded_traffic_is_read_only_for_the_matching_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.md"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    f.write_text(f"kernel_source_hash: {bench.kernel_hash()}\ndram_bytes_per_launch: 446672640\n")
    assert bench.recorded_traffic() == 446672640.0
    f.write_text("kernel_source_hash: 0123456789abcdef\ndram_bytes_per_launch: 446672640\n")
    assert bench.recorded_traffic() is None           # measured on other code
    f.write_text("no figures here\n")
    assert bench.recorded_traffic() is None
    f.unlink()
    assert bench.recorded_traffic() is None           # no summary at all


def _sampler(rows, t0, t1):
    s = bench.ClockSampler("0")
    s.rows = rows
    s.t0, s.t1 = t0, t1
    return s


def _row(sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"2026/12/02 00:00:00.000, {sm}, {smax}, 900.0, {hw}, {hwt}, {swt}, {cap}"


def test_clock_summary_takes_the_timed_region_only():
    rows = [(0.0, _row(2070, 2070)), (0.5, _row(2070, 2070))]                       # before the region
    rows += [(1.0 + 0.1 * i, _row(1600 + i, 2070, cap="Active")) for i in range(5)]  # inside it
    rows += [(9.0, _row(300, 2070, hw="Active"))]                                   # after it
    out = _sampler(rows, 1.0, 1.45).summary()
    assert out["samples"] == 5
    assert out["sm_mhz"] == 1602
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_slowdowns_and_falls_back_to_all_samples():
    rows = [(1.0, _row(1500, 2070, hwt="Active")), (1.1, _row(1700, 2070, swt="Active"))]
    out = _sampler(rows, 5.0, 6.0).summary()          # fewer than 3 samples in the region: all are used
    assert out["samples"] == 2
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert _sampler([], 0.0, 1.0).summary()["reasons"] == ["unsampled"]


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6676.8, "bf16_tflops": 1920.6, '
                                                 '"bf16_tflops_sustained": 1733.0}')
    p = bench.peaks()
    assert p["source"] == "measured" and p["bf16_sus"] == 1733.0 and p["hbm"] == 6676.8


def test_tensor_peak_is_burst_for_short_regions_and_sustained_for_long_ones():
    pk = {"bf16": 1904.0, "bf16_sus": 1709.5, "hbm": 6776.3, "source": "measured"}
    peak, kind = bench.tensor_peak(pk, 0.02)             # 20 steps of about 1 ms
    assert peak == 1904.0 and kind.startswith("bf16 burst")
    peak, kind = bench.tensor_peak(pk, bench.SUSTAINED_REGION_S + 0.5)
    assert peak == 1709.5 and kind.startswith("bf16 sustained")


def test_tensor_peak_follows_the_sampled_clocks():
    pk = {"bf16": 1904.0, "bf16_sus": 1709.5, "hbm": 6776.3, "source": "measured"}
    peak, kind = bench.tensor_peak(pk, 1.1, sm_mhz=1604.5, sm_max_mhz=2070.0)   # capped under load
    assert peak == 1709.5 and "power-capped" in kind
    peak, kind = bench.tensor_peak(pk, 0.02, sm_mhz=2002.0, sm_max_mhz=2070.0)  # full clocks
    assert peak == 1904.0 and kind.startswith("bf16 burst")
    peak, kind = bench.tensor_peak(pk, 0.02, sm_mhz=None, sm_max_mhz=2070.0)    # no samples
    assert peak == 1904.0


def test_lib_peak_takes_the_higher_measured_rate_or_the_fallback():
    assert bench.lib_peak({"burst_tflops": 3400.0, "sustained_tflops": 3350.0}, 1.0) == 3400.0
    assert bench.lib_peak({"burst_tflops": 4900.0, "sustained_tflops": 7000.0}, 1.0) == 7000.0
    assert bench.lib_peak({"error": "no e4m3 GEMM"}, 3808.0) == 3808.0


def test_reference_rows_take_the_whole_batch_when_the_run_fits_the_budget():
    # 3860 tokens/s: a whole 16384-row step takes 4.2 s; 25 steps fit 240 s, 1020 do not
    assert bench.reference_rows(3860.0, 20, 5) == bench.M_TOK
    rows = bench.reference_rows(3860.0, 1000, 20)
    assert rows % 64 == 0 and 64 <= rows < bench.M_TOK
    assert rows / 3860.0 * 1020 <= bench.REFERENCE_BUDGET_S
    assert bench.reference_rows(1.0, 1000, 20) == 64     # never below one 64-row slice

