"""bench.py's clock record, without a GPU: the nvidia-smi samples it parses
give the median loaded SM clock, the throttle reasons seen, and the board
power (median and maximum of the samples, and the enforced limit); a timing
rule rejects runs with hardware or thermal slowdown, so the reasons must be
read exactly."""
import bench

HEAD = "0, {sm}, 2070, {pw}, 0x{act}, {hw}, {hwt}, {swt}, {cap}, 1400.00\n"


def _sampler(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.writelines(lines)
    return s


def test_summary_reads_clocks_reasons_and_power(tmp_path):
    lines = [HEAD.format(sm=sm, pw=pw, act="4", hw="Not Active", hwt="Not Active",
                         swt="Not Active", cap=cap)
             for sm, pw, cap in [(345, 90.5, "Not Active"), (1957, 1100.0, "Active"),
                                 (1980, 1286.2, "Active"), (2070, 700.0, "Not Active")]]
    out = _sampler(tmp_path, lines).summary()
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == 1980.0            # median of the loaded samples (> half of max)
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_max_w"] == 1286.2 and out["power_w"] == 900.0
    assert out["power_limit_w"] == 1400.0
    assert out["samples"] == 4


def test_summary_reports_every_slowdown_reason(tmp_path):
    lines = [HEAD.format(sm=1500, pw=1000, act="8", hw="Active", hwt="Active", swt="Active",
                         cap="Not Active")]
    out = _sampler(tmp_path, lines).summary()
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_summary_without_samples(tmp_path):
    out = _sampler(tmp_path, ["garbage\n"]).summary()
    assert out["reasons"] == ["unsampled"] and out["sm_mhz"] is None
