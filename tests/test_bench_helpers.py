"""Host logic of bench.py that decides what the JSON line reports: the kernel
source hash (source file plus the device headers it includes, in include
order) and the rule that a profile's DRAM traffic is reported only while the
profile was taken on the current source."""
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture
def tree(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text('#include "a.cuh"\n#include <cuda.h>\nint k;\n')
    (csrc / "a.cuh").write_text('#include "b.cuh"\nint a;\n')
    (csrc / "b.cuh").write_text('#include "a.cuh"\nint b;\n')      # cycle: visited once
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_device_headers_in_include_order(tree):
    assert bench._device_headers("k.cu", []) == ["a.cuh", "b.cuh"]


def test_source_hash_covers_included_headers(tree):
    h0 = bench.source_sha1("k.cu")
    assert len(h0) == 12 and h0 == bench.source_sha1("k.cu")
    (tree / "csrc" / "b.cuh").write_text('#include "a.cuh"\nint b2;\n')
    assert bench.source_sha1("k.cu") != h0


def test_profile_traffic_only_for_the_current_source(tree):
    prof = tree / "profiles" / "k.md"
    assert bench.profile_traffic("k.cu", "k.md") is None                  # no summary
    prof.write_text("source_sha1: %s\ndram_bytes_per_launch: 1234567\n" % bench.source_sha1("k.cu"))
    assert bench.profile_traffic("k.cu", "k.md") == 1234567.0
    (tree / "csrc" / "a.cuh").write_text('#include "b.cuh"\nint a_changed;\n')
    assert bench.profile_traffic("k.cu", "k.md") is None                  # source changed since
    prof.write_text("source_sha1: %s\n" % bench.source_sha1("k.cu"))
    assert bench.profile_traffic("k.cu", "k.md") is None                  # no traffic recorded


def test_clock_summary_uses_the_timed_window():
    """Median SM clock and throttle reasons come from the samples taken between
    the two marks (the timed region); unreadable fields are skipped."""
    c = bench.ClockSampler(0)
    row = lambda sm, reasons: [sm, "2070", "900.0", "0x0"] + reasons
    idle = ["Not Active"] * 4
    c.samples = [(0.5, row("1200", ["Active", "Active", "Not Active", "Not Active"])),   # before
                 (1.5, row("2070", idle)), (2.0, row("2010", idle)),
                 (2.5, row("[N/A]", ["Not Active", "Not Active", "Not Active", "Active"])),
                 (3.5, row("900", ["Not Active", "Not Active", "Active", "Not Active"]))]  # after
    c.marks = [1.0, 3.0]
    s = c.summary()
    assert s["sm_mhz"] == 2040.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    c.marks = []                                       # no marks: every sample counts
    assert c.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                                      "sw_thermal_slowdown"]
    assert bench.ClockSampler(0).summary()["reasons"] == ["no samples"]
