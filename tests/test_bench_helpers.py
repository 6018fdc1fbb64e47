"""Host-side checks of the bench's measurement helpers (no GPU): the clock samples kept
for the timed region and the clock-aware roofline arithmetic."""
import bench


def test_clock_summary_keeps_samples_inside_the_timed_region():
    c = bench.ClockSampler(0)
    c.smax = 2070
    c.stamped = [(0.5, 1980, None), (1.0, 2070, ["sw_power_cap"]), (1.5, 2055, None), (2.5, 1400, ["hw_slowdown"])]
    c.t_start, c.t_end = 0.9, 2.0
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == (2070 + 2055) / 2
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070


def test_clock_aware_roofline_arithmetic():
    pk = {"bf16_tflops": 1909.9}
    r = bench.clock_aware_roofline(1350.0, pk, {"sm_mhz": 2070.0}, 152, 1477.0)
    at_clock = 152 * 8192 * 2070.0e6 / 1e12  # one 128x128x16 MMA per 64 cycles per SM
    assert abs(r["peak_at_kernel_clock"] - at_clock) < 1e-6
    assert abs(r["frac_of_clock_peak"] - 1350.0 / at_clock) < 1e-12
    assert abs(r["frac_clock_scaled"] - 1350.0 * 1477.0 / 2070.0 / 1909.9) < 1e-12
    assert bench.clock_aware_roofline(1350.0, pk, {"sm_mhz": None}, 152, 1477.0) == {}
    assert "frac_clock_scaled" not in bench.clock_aware_roofline(1350.0, pk, {"sm_mhz": 2070.0}, 152, None)

