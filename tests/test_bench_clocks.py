"""The bench keeps a timed run unless its clock record shows a hardware or thermal
slowdown or a clock stuck well below maximum with no reason (then it measures once
more); a power-cap slowdown is kept and reported."""
import bench


def test_power_cap_is_kept():
    assert not bench.clocks_suspect({"sm_mhz": 1640, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"]})


def test_hardware_and_thermal_slowdowns_are_remeasured():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_suspect({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": [r, "sw_power_cap"]})


def test_a_clock_stuck_low_without_reason_is_remeasured():
    assert bench.clocks_suspect({"sm_mhz": 1000, "sm_max_mhz": 2070, "reasons": []})
    assert not bench.clocks_suspect({"sm_mhz": 1900, "sm_max_mhz": 2070, "reasons": []})


def test_no_record_is_kept():
    assert not bench.clocks_suspect(None)
    assert not bench.clocks_suspect({"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
