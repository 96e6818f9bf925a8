"""The benchmark's clock record: nvidia-smi CSV samples taken during the timed
region become the ``clocks`` object of the JSON line (median SM clock, the
maximum clock, every throttle reason seen).  Parsed here from a written CSV in
nvidia-smi's format, no GPU involved."""
import time

import bench

FMT = "%Y/%m/%d %H:%M:%S"


def _line(t, uuid, sm, reasons=("Not Active",) * 4, sm_max=2070):
    ts = time.strftime(FMT, time.localtime(int(t))) + f".{int((t % 1) * 1000):03d}"
    return f"{ts}, {uuid}, {sm}, {sm_max}, 912.40, 0x0000000000000000, " + ", ".join(reasons) + "\n"


def _sampler(tmp_path, lines, uuid="GPU-1234"):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(lines))
    s = bench.ClockSampler(uuid)
    s.path = str(path)
    return s


def test_median_clock_and_no_reasons_in_the_window(tmp_path):
    t0 = float(int(time.time())) + 0.5
    lines = [_line(t0 + 0.1 * i, "GPU-1234", sm) for i, sm in enumerate((2070, 2055, 2070, 1980, 2070))]
    lines.append(_line(t0 + 0.2, "GPU-9999", 600))  # another GPU's line: ignored
    out = _sampler(tmp_path, lines).summary(t0, t0 + 0.4)
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == [] and out["samples"] == 5 and not out["nearest_only"]


def test_throttle_reasons_are_reported_by_name(tmp_path):
    t0 = float(int(time.time())) + 0.5
    active = ("Not Active", "Not Active", "Active", "Active")  # hw, hw thermal, sw thermal, sw power cap
    lines = [_line(t0, "GPU-1234", 1900), _line(t0 + 0.1, "GPU-1234", 1890, active)]
    out = _sampler(tmp_path, lines).summary(t0, t0 + 0.1)
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1895


def test_nearest_sample_when_none_falls_in_the_window(tmp_path):
    t0 = float(int(time.time())) + 0.5
    lines = [_line(t0 - 5.0, "GPU-1234", 1500), _line(t0 + 5.0, "GPU-1234", 2070)]
    out = _sampler(tmp_path, lines).summary(t0 + 3.0, t0 + 3.2)
    assert out["nearest_only"] and out["samples"] == 0 and out["sm_mhz"] == 2070


def test_no_samples_reads_as_unavailable(tmp_path):
    out = _sampler(tmp_path, []).summary(0.0, 1.0)
    assert out["reasons"] == ["unavailable"] and out["sm_mhz"] is None
