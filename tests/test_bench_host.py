"""bench.py's host logic on the CPU: the committed ncu traffic figure is used only while the
kernel sources hash to the digest recorded beside it; the clock summary reads nvidia-smi's CSV
(median SM clock, throttle reasons); the whole-job rate counts every rank's units."""
import os
import subprocess
import sys

import pytest

import bench


def test_recorded_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    digest = bench.kernel_source_digest("gemm1_swiglu")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemm1_swiglu_fake.ncu.txt").write_text(
        f"# comment lines: ignored\n# kernel_sources: not this one\nkernel_sources: {digest}\n"
        "dram_bytes_per_launch: 123456789\n")
    (prof / "gemm1_swiglu_stale.ncu.txt").write_text("kernel_sources: 0000000000000000\ndram_bytes_per_launch: 5\n")
    real_join = os.path.join

    def join(*a):  # the profiles folder from tmp_path, the kernel sources from the repository
        if len(a) >= 2 and a[0] == bench.ROOT and a[1] == "profiles":
            return real_join(str(tmp_path), *a[1:])
        return real_join(*a)

    monkeypatch.setattr(bench.os.path, "join", join)
    assert bench.recorded_traffic("fake", "gemm1_swiglu") == 123456789.0
    assert bench.recorded_traffic("stale", "gemm1_swiglu") is None
    assert bench.recorded_traffic("missing", "gemm1_swiglu") is None


def test_committed_traffic_matches_the_current_sources():
    """The large_e64 figure the benchmark prints is the committed one, taken on these sources."""
    t = bench.recorded_traffic("large_e64", "gemm1_swiglu")
    assert t is not None and 3.0e9 < t < 6.0e9


def test_clock_summary_reads_median_and_reasons(tmp_path):
    s = bench.ClockSampler(0)
    f = tmp_path / "clocks.csv"
    rows = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1600, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1650, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbage line"]
    f.write_text("\n".join(rows) + "\n")
    s.file = open(f, "a")
    s.proc = object()
    out = s.summary()
    assert out["sm_mhz"] == 1650.0 and out["sm_max_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]


def test_throughput_counts_every_rank():
    assert bench.throughput(4096, 10, 1, 50.0) == pytest.approx(4096 * 10 / 0.05)
    assert bench.throughput(4096, 10, 4, 50.0) == pytest.approx(4 * 4096 * 10 / 0.05)


def test_help_lists_the_modes():
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--help"], capture_output=True,
                         text=True, timeout=120).stdout
    for flag in ("--gpus", "--steps", "--warmup", "--impl", "--workload", "--train", "--perf-model", "--sweep",
                 "--ep-stage"):
        assert flag in out
