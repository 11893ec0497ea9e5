"""Host logic of bench.py that needs no GPU: the clock-sample window filter
(samples are kept only when stamped inside the timed region; the nearest
one stands in, with samples = 0, when the region is shorter than the
sampling period) and throttle-reason collection."""
import datetime

import bench


def _line(t, sm, mx, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return (f"{ts}, 0, {sm}, {mx}, 900.00, 0x0000000000000000, Not Active, "
            f"{thermal}, Not Active, {power_cap}\n")


def test_window_keeps_only_inside_samples():
    t = 1_800_000_000.0
    lines = [_line(t, 1000, 2070), _line(t + 0.1, 2070, 2070),
             _line(t + 0.15, 2050, 2070, power_cap="Active"), _line(t + 0.5, 900, 2070)]
    got = bench.parse_clock_samples(lines, t + 0.05, t + 0.2)
    assert got["samples"] == 2
    assert got["sm_mhz"] == 2060
    assert got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]


def test_short_region_takes_nearest_sample():
    t = 1_800_000_000.0
    lines = [_line(t, 1500, 2070), _line(t + 0.05, 2070, 2070, thermal="Active")]
    got = bench.parse_clock_samples(lines, t + 0.04, t + 0.045)
    assert got["samples"] == 0
    assert got["sm_mhz"] == 2070 and got["reasons"] == ["hw_thermal_slowdown"]


def test_garbage_lines_ignored():
    assert bench.parse_clock_samples(["", "bad line\n"], 0.0, 1.0) is None


def test_sampled_launches_rotate_through_the_layers():
    got = bench.sampled_launches(64, 32, 1)
    assert len(got) == 64
    assert [l for _, l in got] == [s % 32 for s in range(64)]
    per_layer = {}
    for _, l in got:
        per_layer[l] = per_layer.get(l, 0) + 1
    assert sorted(per_layer) == list(range(32)) and set(per_layer.values()) == {2}
    two = bench.sampled_launches(3, 32, 2)
    assert two == [(0, 0), (0, 1), (1, 2), (1, 3), (2, 4), (2, 5)]
    assert bench.sampled_launches(3, 1, 1) == [(0, 0), (1, 0), (2, 0)]
    assert len(bench.sampled_launches(5, 3, 4)) == 15
