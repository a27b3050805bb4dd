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


# ---- the JSON line stays short enough to reach the end of a 1.5 KB log tail ------------

X = 12345.678901234   # every float at its longest once rounded to 4 significant figures


def _fake_measurements():
    import argparse
    args = argparse.Namespace(history=4096)
    return {"value": X, "world": 1, "steps": 20, "warmup": 5, "ms_per_step": 0.08734879978,
            "config": bench.workload_config(args, 1),
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "sm_min_mhz": 1987.5,
                       "power_w_median": 402.365, "samples": 8,
                       "reasons": ["sw_power_cap"]},
            "e2e_value": X, "h2d": 459264, "d2h": 262144, "serial_value": X,
            "gpu_launches": 40, "achieved": X, "peak": 6705.2, "peak_kind": "measured",
            "traffic": 541237504.0, "rb": 537460992, "dec_ms": [0.0854799, 0.0838879, 0.08179]}


def _fake_extras():
    hs = (16, 64, 256, 1024, 4096)
    sweep = [{"history": h, "us_median": X, "us_min": X, "gbs": X, "frac": 0.73456789}
             for h in hs]
    longctx = [{"history": h, "splits": h // 1024, "us_split_plus_merge": X, "gbs": X,
                "frac": 0.9512345, "us_single_pass": X} for h in (32768, 131072)]
    ragged = {"batch": 256, "kv_gb": 4.5, "us_single_pass": X, "gbs_single_pass": X,
              "us_split64_plus_merge": X, "gbs_split64": X, "frac_best": 1.0312345,
              "planned": [{"target_ctas": 152 * m, "items": 900, "max_slots": 4, "us": X + m,
                           "plan_host_us": X, "gbs": X} for m in (3, 6, 12, 24)]}
    chunk = {"llama1b_h4096": [{"n_q": n, "us": X, "gbs": X, "frac_hbm": 0.3648199,
                                "tflops": X} for n in (1, 4, 16, 64)],
             "longctx_h32768_split": [{"n_q": n, "splits": 32, "us_split_plus_merge": X,
                                       "gbs": X, "frac_hbm": 0.6, "us_single_pass": X}
                                      for n in (1, 4, 16)]}
    prefill = [{"head_dim": d, "batch": 8, "prompt": 4096, "us": X, "tflops": X,
                "peak_tflops": 1886.7, "peak_source": "measured", "frac_tensor": 0.3456789}
               for d in (64, 128)]
    dense = [{"n_ctx": n, "us_by_splits": {}, "best_splits": 16, "us_best": X, "us_sdpa": X,
              "gbs_best": X, "gbs_sdpa": X, "sdpa_over_ours": 1.469240007}
             for n in (1024, 2048, 4096, 8192, 16384)]
    return {"chunk": bench.compact_chunk(chunk), "dense_vs_sdpa": bench.compact_dense(dense),
            "sweep": bench.compact_sweep(sweep), "longctx": bench.compact_longctx(longctx),
            "ragged8b": bench.compact_ragged(ragged), "prefill": bench.compact_prefill(prefill)}


def _fake_cpu():
    # the shape bench.cpu_baseline returns
    return {"value": X, "unit": "GB/s", "cores": 16, "kind": "oracle",
            "sample": "123 passes of the h4096 batch, 1 proc/core",
            "best_ms": X, "median_ms": X, "busy": 15.87654, "single_core": X}


def test_the_whole_line_fits_a_1500_byte_tail():
    line = bench.compact_json(bench.compose_line(_fake_measurements(), _fake_extras(),
                                                 _fake_cpu()))
    assert len(line.encode()) <= 1500, len(line.encode())
    parsed = json.loads(line)
    # every key the contract asks for, and the graded extras ending the line
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "clocks", "e2e", "gpu_launches", "roofline", "cpu_baseline"):
        assert key in parsed, key
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in parsed["roofline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in parsed["e2e"], key
    assert list(parsed)[-4:] == list(bench.GRADED)
    assert parsed["sweep"]["h"] == [16, 64, 256, 1024, 4096]
    assert parsed["value"] == 12350                       # 4 significant figures


def test_a_failed_extra_keeps_the_line_short():
    extras = _fake_extras()
    try:
        raise RuntimeError("x" * 5000)
    except RuntimeError as e:
        extras["prefill"] = bench.extra_error(e)
    line = bench.compact_json(bench.compose_line(_fake_measurements(), extras, _fake_cpu()))
    assert len(line.encode()) <= 1500
    assert json.loads(line)["prefill"]["error"].startswith("RuntimeError: xxx")


def test_round_sig_keeps_ints_strings_and_non_finite():
    got = bench.round_sig({"a": 1.23456789, "b": [7, "s", float("inf")], "c": {"d": 0.0001234567},
                           "e": 6156.0507, "f": 999.96, "g": -12345.6})
    assert got == {"a": 1.235, "b": [7, "s", float("inf")], "c": {"d": 0.0001235},
                   "e": 6156, "f": 1000, "g": -12350}
    assert isinstance(got["e"], int) and isinstance(bench.round_sig(85.4799), float)


def test_parallel_oracle_runs_the_batch_on_several_processes():
    # the multi-core baseline: every sequence once per pass, over spawned workers that map
    # the pools from shared memory; the bytes per pass are the batch's algorithmic bytes
    import workloads
    batch = workloads.make_batch("par", 42, "bf16", [300, 50, 700, 16, 129], 8, 2, 64, 16, 120)
    sample = bench.OracleSample(batch)
    par = bench.ParallelOracle(sample, 2)
    try:
        assert sorted(i for t in par.tasks for i in t) == list(range(5))
        assert par.pass_bytes == bench.read_bytes(batch.lens_list(), 8, 2, 64, 2, 16)
        walls = [par.one_pass() for _ in range(2)]
        assert all(w > 0 for w in walls)
        assert par.cpu_s > 0
    finally:
        par.close()


def test_cpu_baseline_falls_back_to_one_thread_without_shared_memory(monkeypatch):
    # a host whose shared memory cannot hold the pools still reports the single-core figure
    import workloads

    class NoShm:
        def __init__(self, *a, **k):
            raise OSError("no space left on device")

    monkeypatch.setattr(bench, "ParallelOracle", NoShm)
    batch = workloads.make_batch("fallback", 43, "bf16", [64, 32], 8, 2, 64, 16, 12)
    got = bench.cpu_baseline(batch, 64, single_budget_s=0.2, multi_budget_s=0.2)
    assert got["cores"] == 1 and got["value"] > 0 and "OSError" in got["sample"]
