"""The benchmark's run records on CPU.  The clock record: nvidia-smi samples
(csv, no header, no units) are reduced to the median SM clock under load, the
maximum clock and the throttle reasons seen, so that a throttled or
clock-locked run can be recognised and rejected.  The roofline traffic: the
committed ncu figure is used only while the kernel it was measured on is
unchanged."""
import bench

CLEAN = "0, 2070, 2070, 880.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"


def _summary(tmp_path, lines):
    s = bench.ClockSampler(0)
    p = tmp_path / "clocks.csv"
    p.write_text("".join(lines))
    s.path = str(p)
    return s.summary()


def test_clean_run(tmp_path):
    got = _summary(tmp_path, [CLEAN] * 5)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}


def test_reasons_and_median(tmp_path):
    lines = [CLEAN,
             "0, 1980, 2070, 1390.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
             "0, 1500, 2070, 900.00, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n",
             "0, 2070, 2070, 900.00, 0x0000000000000000, Not Active, Active, Active, Not Active\n"]
    got = _summary(tmp_path, lines)
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert got["sm_mhz"] == 2025.0 and got["sm_max_mhz"] == 2070.0 and got["samples"] == 4


def test_clock_stuck_low_without_a_reason_is_visible(tmp_path):
    # a leftover clock lock shows as a median far below the maximum with no reason active
    got = _summary(tmp_path, ["0, 1200, 2070, 600.00, 0x0000000000000000, Not Active, Not Active, Not Active, "
                              "Not Active\n"] * 3)
    assert got["reasons"] == [] and got["sm_mhz"] == 1200.0 and got["sm_max_mhz"] == 2070.0


def test_malformed_lines_are_skipped_and_no_samples_is_none(tmp_path):
    got = _summary(tmp_path, ["garbage\n", "0, [N/A], 2070, 1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
                              CLEAN])
    assert got["samples"] == 1
    assert _summary(tmp_path, ["garbage\n"]) is None


def test_roofline_traffic_is_tied_to_the_kernel_source(tmp_path, monkeypatch):
    # the committed ncu traffic is reported only while the fingerprint kernel's source is the one it
    # was measured on, and only for the workload it was scaled to
    import json
    import os
    import shutil
    full = bench.scan_traffic(24)
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "fp_scan_traffic.json")))
    assert full == d["dram_bytes_per_launch"] * d["scale_to_full"]
    assert bench.scan_traffic(0) is None
    fake = tmp_path / "root"
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), fake / "profiles")
    csrc = fake / "silent_corruption_checksums_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = open(os.path.join(bench.ROOT, "silent_corruption_checksums_gb300", "csrc", "sdc_fp.cu"), "rb").read()
    (csrc / "sdc_fp.cu").write_bytes(src)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.scan_traffic(24) == full
    (csrc / "sdc_fp.cu").write_bytes(src + b"\n// changed\n")
    assert bench.scan_traffic(24) is None
