"""The benchmark's summary of the SM clocks sampled during the timed region
(CPU only).

A measurement taken under a hardware or thermal slowdown, or with the clocks
stuck low, is not valid, so the reasons nvidia-smi reports active must come
through exactly.  The lines below have the layout of
`nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`.
"""
import bench


def _line(sm, smax, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active",
          mask="0x0000000000000000"):
    return f"{sm}, {smax}, 812.40, {mask}, {hw}, {hw_th}, {sw_th}, {cap}\n"


def test_median_clock_max_clock_and_power_cap():
    lines = [_line(1500, 2032, cap="Active", mask="0x0000000000000004"), _line(1582, 2032),
             _line(1700, 2032)]
    s = bench.summarise_clock_samples(lines)
    assert s == {"sm_mhz": 1582.0, "sm_max_mhz": 2032.0, "samples": 3, "reasons": ["sw_power_cap"]}


def test_every_slowdown_reason_is_reported():
    lines = [_line(900, 2032, hw="Active"), _line(950, 2032, hw_th="Active"),
             _line(1000, 2032, sw_th="Active")]
    s = bench.summarise_clock_samples(lines)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 950.0


def test_partial_and_unavailable_samples_are_skipped():
    lines = [_line(1600, 2032), "1610, 2032, 80", _line("[N/A]", 2032, hw="Active"), "\n",
             _line(1620, "[N/A]", cap="Active")]
    s = bench.summarise_clock_samples(lines)
    # only the first line is a complete sample; the skipped ones add no reason
    assert s == {"sm_mhz": 1600.0, "sm_max_mhz": 2032.0, "samples": 1, "reasons": []}


def test_no_samples_gives_none():
    assert bench.summarise_clock_samples([]) is None
    assert bench.summarise_clock_samples(["garbage\n"]) is None


def test_only_samples_inside_the_timed_region_count():
    import datetime
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    def stamped(sm, dt_ms, cap="Not Active"):
        t = base + datetime.timedelta(milliseconds=dt_ms)
        return _line(sm, 2032, cap=cap).rstrip("\n") + ", " + t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3] + "\n"
    lines = [stamped(2032, 0), stamped(1500, 100, cap="Active"), stamped(1600, 120), stamped(1700, 140),
             stamped(1000, 400, cap="Active")]
    t0 = (base + datetime.timedelta(milliseconds=90)).timestamp()
    t1 = (base + datetime.timedelta(milliseconds=150)).timestamp()
    s = bench.summarise_clock_samples(lines, t0, t1)
    # the idle sample before the region and the one after it are left out
    assert s == {"sm_mhz": 1600.0, "sm_max_mhz": 2032.0, "samples": 3, "reasons": ["sw_power_cap"]}
    assert bench.summarise_clock_samples(lines, t1 + 1.0, t1 + 2.0) is None
