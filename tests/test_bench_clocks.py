"""The bench's clock record on CPU: nvidia-smi sample lines (made up here, in
the CSV form the sampler asks for) are parsed, and the summary keeps only
the samples stamped inside the loaded window around the timed region, with
the throttle reasons of those samples alone.  No GPU and no nvidia-smi."""
import datetime

import bench


def _line(t, sm, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join(["0", str(sm), "2070", "900.0", "0x0", *flags, stamp]) + "\n"


def _sampler(tmp_path, lines, t0=None, t1=None):
    clk = bench.ClockSampler(0)
    clk.path = str(tmp_path / "clocks.csv")
    with open(clk.path, "w") as f:
        f.writelines(lines)
    clk.t_start, clk.t_end = t0, t1
    return clk


def test_only_samples_inside_the_window_count(tmp_path):
    base = 1_800_000_000.0
    lines = [_line(base + 0.0, 1200, {"sw_thermal_slowdown"}),  # idle, before the window
             _line(base + 0.5, 2070), _line(base + 0.6, 2070), _line(base + 0.7, 2055, {"sw_power_cap"}),
             _line(base + 2.0, 1000, {"hw_slowdown"})]  # after the window
    s = _sampler(tmp_path, lines, base + 0.45, base + 1.2).summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["window_s"] == 0.75


def test_without_a_window_every_sample_counts(tmp_path):
    base = 1_800_000_000.0
    lines = [_line(base, 2070), _line(base + 0.1, 1900, {"hw_thermal_slowdown"})]
    s = _sampler(tmp_path, lines).summary()
    assert s["samples"] == 2
    assert s["reasons"] == ["hw_thermal_slowdown"]
    assert "window_s" not in s


def test_unreadable_stamps_keep_every_sample(tmp_path):
    lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active, n/a\n",
             "0, 2000, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active, n/a\n"]
    s = _sampler(tmp_path, lines, 0.0, 1.0).summary()
    assert s["samples"] == 2
    assert s["sm_mhz"] == 2035


def test_no_samples_reads_unavailable(tmp_path):
    s = _sampler(tmp_path, ["garbage\n"]).summary()
    assert s["reasons"] == ["unavailable"]
