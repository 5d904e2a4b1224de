"""The bench's clock record: how nvidia-smi samples become the JSON line's
`clocks` object (median SM clock under load, the highest reported maximum,
and every throttle reason seen active), from samples inside the timed region
when there are any.  No GPU: the sampler is fed lines in nvidia-smi's CSV
format (index, clocks.sm, clocks.max.sm, power.draw, reasons.active,
hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap)."""
import bench


def _line(sm, sm_max, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    return f"0, {sm}, {sm_max}, 1012.5, 0x0000000000000000, {hw}, {hw_th}, {sw_th}, {cap}"


def _sampler(samples):
    s = bench.ClockSampler(0)
    s.lines = list(samples)
    return s


def test_median_and_max_from_the_timed_region_only():
    s = _sampler([(0.5, _line(1200, 2070, hw="Active")),     # before the timed region
                  (1.0, _line(2070, 2070)), (1.5, _line(2040, 2070)), (2.0, _line(1995, 2070)),
                  (3.5, _line(900, 2100, sw_th="Active"))])  # after it
    c = bench.ClockSampler.summary(s, 1.0, 2.0)
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == [] and c["samples"] == 3 and c["samples_in_timed_region"] == 3


def test_reasons_active_inside_the_region_are_reported():
    s = _sampler([(1.0, _line(2070, 2070, cap="Active")), (1.2, _line(1800, 2070, hw_th="Active")),
                  (1.4, _line(2070, 2070))])
    c = s.summary(0.9, 1.5)
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert c["sm_mhz"] == 2070.0


def test_no_sample_inside_falls_back_to_all_and_malformed_lines_are_skipped():
    s = _sampler([(0.1, "garbage"), (0.2, "0, [N/A], 2070, 1, 0, Not Active, Not Active, Not Active, Not Active"),
                  (0.3, _line(1500, 2070)), (0.4, _line(1700, 2070))])
    c = s.summary(5.0, 6.0)
    assert c["samples"] == 2 and c["samples_in_timed_region"] == 0
    assert c["sm_mhz"] == 1600.0


def test_no_samples_at_all():
    c = _sampler([]).summary(0.0, 1.0)
    assert c["sm_mhz"] is None and c["reasons"] == ["no samples"] and c["samples"] == 0
