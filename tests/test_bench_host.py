"""Host-side logic of the benchmark that decides what a reported number
means: the clock record a run is accepted or rejected on, the algorithmic
bytes the HBM roofline fractions divide, and the rule that a recorded DRAM
traffic figure is reported only for the kernel source it was captured on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _line(sm, smax, util, power, active, hw, hwt, swt, pcap):
    return f"{sm}, {smax}, {util}, {power}, {active}, {hw}, {hwt}, {swt}, {pcap}\n"


def test_clock_summary_median_under_load_and_reasons():
    na, ac = "Not Active", "Active"
    lines = [
        _line(1000, 2070, 0, 150.0, "0x0", na, na, na, na),        # idle: not counted for the median
        _line(1950, 2070, 100, 1200.0, "0x4", na, na, na, ac),     # power cap under load
        _line(1965, 2070, 100, 1250.0, "0x0", na, na, na, na),
        _line(1980, 2070, 99, 1300.0, "0x0", na, na, na, na),
        "garbage line\n",
        _line(900, 2070, 0, 140.0, "0x8", ac, na, na, na),         # a slowdown while idle: not counted
    ]
    d = bench.summarize_clock_samples(lines)
    assert d["sm_mhz"] == 1965.0
    assert d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"]
    assert d["samples"] == 5 and d["samples_under_load"] == 3


def test_clock_summary_reports_each_slowdown_under_load():
    na, ac = "Not Active", "Active"
    for i, name in enumerate(bench.CLOCK_REASONS):
        flags = [na] * 4
        flags[i] = ac
        d = bench.summarize_clock_samples([_line(1500, 2070, 100, 900.0, "0x1", *flags)])
        assert d["reasons"] == [name]


def test_clock_summary_without_samples():
    assert bench.summarize_clock_samples([])["reasons"] == ["no samples"]
    # all idle: the median falls back to every sample
    d = bench.summarize_clock_samples([_line(1200, 2070, 0, 100.0, "0x0", *(["Not Active"] * 4))])
    assert d["sm_mhz"] == 1200.0 and d["samples_under_load"] == 1


def test_algorithmic_bytes_of_the_hbm_bound_workloads():
    """A + B + C once, plus the int4 scales and zero points: the figures the
    skinny and int4 roofline fractions divide."""
    by_name = {c.name: c for c in wl.WORKLOADS}
    skinny = [c for c in by_name.values() if c.M == 64 and c.N == 4096 and c.K == 16384]
    int4 = [c for c in by_name.values() if c.b_dtype == wl.INT4]
    assert len(skinny) == 1 and len(int4) == 1
    s, q = skinny[0], int4[0]
    assert bench.algorithmic_bytes(s) == 64 * 16384 * 2 + 4096 * 16384 * 2 + 64 * 4096 * 2 == 136839168
    groups = 16384 // 128
    expect = 16 * 16384 * 2 + 16384 * 16384 // 2 + 16 * 16384 * 2 + 16384 * groups * 2 * 2
    assert bench.algorithmic_bytes(q) == expect == 143654912


def test_recorded_traffic_only_for_the_current_source(tmp_path, monkeypatch):
    """profiles/traffic.json's figure is reported only while the hash of the
    headline kernel's sources equals the one it was captured on."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        with open(os.path.join(ROOT, rel), "rb") as f:
            dst.write_bytes(f.read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_hash()
    (prof / "traffic.json").write_text(json.dumps({"w": {"source_sha": sha, "dram_bytes_per_launch": 123}}))
    assert bench.recorded_traffic("w") == 123
    assert bench.recorded_traffic("other") is None
    # any edit of a listed source invalidates it
    first = tmp_path / bench.KERNEL_SOURCES[0]
    first.write_bytes(first.read_bytes() + b"\n")
    assert bench.recorded_traffic("w") is None
