"""bench.py's clock record: only nvidia-smi samples that arrived while the
timed steps ran count, and every throttle reason seen among them is listed."""
import bench


def _line(sm, reasons=("Not Active",) * 4):
    # index, clocks.sm, clocks.max.sm, power.draw, active mask, 4 reasons
    return ", ".join(["0", str(sm), "2070", "1200.5", "0x0", *reasons])


def test_summary_keeps_only_samples_inside_the_window():
    s = bench.ClockSampler(0)
    s.lines = [(0.0, _line(2070)), (0.1, _line(2070)),          # idle, before the steps
               (1.00, _line(1890)), (1.02, _line(1875)), (1.05, _line(1900)),
               (2.0, _line(2070))]                              # idle, after
    c = s.summary(0.9, 1.1)
    assert c["samples"] == 3 and c["sm_mhz"] == 1890 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == []
    assert s.summary()["samples"] == 6


def test_summary_lists_throttle_reasons_in_the_window_only():
    s = bench.ClockSampler(0)
    cap = ("Not Active", "Not Active", "Not Active", "Active")
    hot = ("Not Active", "Active", "Not Active", "Not Active")
    s.lines = [(0.5, _line(1500, hot)), (1.0, _line(1700, cap)), (1.01, "garbled"),
               (1.02, _line(1710))]
    c = s.summary(0.9, 1.1)
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 2


def test_summary_without_samples():
    s = bench.ClockSampler(0)
    c = s.summary(0.0, 1.0)
    assert c["samples"] == 0 and c["sm_mhz"] is None
