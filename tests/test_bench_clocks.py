"""The bench's clocks record, parsed from nvidia-smi CSV lines as the sampler receives them: the
median SM clock under load, the maximum clock, and every throttle reason that was active in any
sample (a run that saw a thermal or hardware slowdown must say so)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, reasons=()):
    flags = ["Active" if n in reasons else "Not Active" for n in bench.ClockSampler.NAMES]
    return ", ".join(["0", str(sm), "2070", "900.00", "0x0000000000000000"] + flags)


def test_median_under_load_and_max():
    out = "\n".join(_line(s) for s in (2070, 2055, 2040, 345))   # the idle sample is left out
    r = bench.parse_clocks(out)
    assert r["sm_mhz"] == 2055 and r["sm_max_mhz"] == 2070 and r["reasons"] == [] and r["samples"] == 4


def test_any_active_reason_is_reported():
    out = "\n".join([_line(2070), _line(1980, ("sw_power_cap",)), _line(1500, ("hw_thermal_slowdown",))])
    assert bench.parse_clocks(out)["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_malformed_and_empty_output():
    assert bench.parse_clocks("")["reasons"] == ["no samples"]
    assert bench.parse_clocks("garbage\n1, 2\n0, [N/A], [N/A], 1, 0, a, b, c, d")["sm_mhz"] is None
