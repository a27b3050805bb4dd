"""bench.py's host-side pieces that need no GPU: the roofline denominators,
the ncu traffic figure it reports beside the achieved bandwidth, and the
clock sampler (against a stand-in nvidia-smi that prints fixed rows)."""

import json
import os
import sys
import tempfile
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_peaks_fall_back_without_a_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    assert bench.measured_bf16_tflops() == (1900.0, "fallback")


def test_peaks_come_from_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 7012.5, "bf16_tflops": 1911.0, "bf16_tflops_sustained": 1702.0,
         "clocks": {"sm_mhz": 2070}}))
    assert bench.measured_peaks() == (7012.5, "measured")
    # the burst figure: the prefill kernel is timed alone, not inside a long step
    assert bench.measured_bf16_tflops() == (1911.0, "measured")


def test_unreadable_peaks_file_falls_back(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.measured_peaks()[1] == "fallback"
    assert bench.measured_bf16_tflops()[1] == "fallback"


def test_committed_profile_describes_the_current_read_kernel():
    # the traffic figure is reported only while the profile's source hash matches the
    # kernel source it was captured from
    traffic = bench.profiled_traffic()
    assert traffic is not None, "profile's source_sha no longer matches the read kernel"
    algorithmic = bench.read_bytes([4096] * 64, 32, 8, 64, 2, 16)
    assert algorithmic == 537_460_992
    assert 1.0 <= traffic / algorithmic < 1.05


def test_stale_profile_reports_no_traffic(monkeypatch):
    monkeypatch.setattr(bench, "source_sha", lambda: "0" * 16)
    assert bench.profiled_traffic() is None


@pytest.mark.parametrize("lens,want", [
    ([1], 1 * 8 * 64 * 2 * 2 + 2 * 32 * 64 * 2 + 4 * 1 + 4),
    ([16, 17], 33 * 8 * 64 * 2 * 2 + 2 * 2 * 32 * 64 * 2 + 4 * 3 + 4 * 2),
])
def test_read_bytes_counts_kv_q_out_table_and_lengths(lens, want):
    assert bench.read_bytes(lens, 32, 8, 64, 2, 16) == want


_FAKE_SMI = """#!/bin/sh
# stands in for nvidia-smi --query-gpu ... -lms 200: prints fixed samples, then waits
cat <<'ROWS'
0, 2070, 2070, 480.25, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
0, 2055, 2070, 501.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active
garbage line
0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active
0, 1980, 2070, 510.50, 0x0000000000000008, Active, Not Active, Not Active, Not Active
ROWS
exec sleep 30
"""


def test_clock_sampler_reports_the_median_and_every_active_reason(monkeypatch, tmp_path):
    smi = tmp_path / "nvidia-smi"
    smi.write_text(_FAKE_SMI)
    smi.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    monkeypatch.setattr(tempfile, "tempdir", str(tmp_path))
    s = bench.ClockSampler(0)
    s.start()
    assert s.path.startswith(str(tmp_path))
    got = s.stop()
    assert got["samples"] == 3                      # the malformed rows are skipped
    assert got["sm_mhz"] == 2055.0 and got["sm_min_mhz"] == 1980.0
    assert got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert not list(tmp_path.glob("clocks_*.csv"))  # the sample file is removed


def test_clock_sampler_without_nvidia_smi(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))       # an empty directory: no nvidia-smi
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_oracle_sample_counts_bytes_and_runs_on_one_thread():
    import workloads
    batch = workloads.make_batch("cpu_sample", 40, "bf16", [300, 50, 4096], 32, 8, 64, 16, 300)
    sample = bench.OracleSample(batch)
    t, nb, n = sample.run(60.0, 2, first=1)
    assert n == 2 and t > 0
    assert nb == bench.read_bytes([50], 32, 8, 64, 2, 16) + bench.read_bytes([4096], 32, 8, 64, 2,
                                                                             16)
    # the ratio over a longer run, once the threads of the batch draw have gone idle
    sample.cpu_s = sample.wall_s = 0.0
    time.sleep(0.2)
    sample.run(60.0, 6, first=2)
    assert 0 < sample.cpu_per_wall() <= 1.5


class _ScriptedClock:
    """Stands in for the time module: each perf_counter() call is one second after the
    last; process_time() advances 2.5 s per call."""

    def __init__(self):
        self.wall = -1.0
        self.cpu = -2.5

    def perf_counter(self):
        self.wall += 1.0
        return self.wall

    def process_time(self):
        self.cpu += 2.5
        return self.cpu


def test_oracle_sample_stops_at_its_budget_on_a_scripted_clock(monkeypatch):
    import workloads
    batch = workloads.make_batch("clock", 41, "f32", [20, 9, 33, 5], 4, 2, 8, 4, 40)
    sample = bench.OracleSample(batch)
    monkeypatch.setattr(bench, "time", _ScriptedClock())
    # start at 0; the budget check after sequences 1, 2, 3 reads 1, 2, 3 s: 3 > 2.5 stops it,
    # and the final reading (4 s) is the wall time returned
    t, nb, n = sample.run(2.5, 64, first=1)
    assert (t, n) == (4.0, 3)
    assert nb == sum(bench.read_bytes([x], 4, 2, 8, 4, 4) for x in (9, 33, 5))
    assert sample.cpu_per_wall() == pytest.approx(2.5 / 4.0, abs=0.01)   # rounded to 0.01
    # a count limit ends the run before the budget does
    t, nb, n = sample.run(100.0, 2, first=0)
    assert n == 2 and nb == sum(bench.read_bytes([x], 4, 2, 8, 4, 4) for x in (20, 9))
