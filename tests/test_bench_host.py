"""Host-side logic of bench.py that needs no GPU: the clock windows built
from timestamped nvidia-smi samples, and the roofline peaks of each leg."""
import types

import bench


def _sampler_with(rows):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = object()  # a sampler that ran
    s.rows = rows
    return s


def test_clock_window_keeps_only_samples_inside_the_load_windows():
    rows = [(0.5, 1500.0, 2070.0, 300.0, set()),            # before: idle
            (1.1, 2070.0, 2070.0, 900.0, set()),            # inside window 1
            (1.2, 2060.0, 2070.0, 950.0, {"sw_power_cap"}),  # inside window 1
            (2.0, 800.0, 2070.0, 200.0, {"hw_slowdown"}),    # between windows
            (3.5, 2070.0, 2070.0, 1000.0, set())]           # inside window 2
    s = _sampler_with(rows)
    w = s.window([(1.0, 1.5), (3.0, 4.0)])
    assert w["samples_under_load"] == 3
    assert w["sm_mhz"] == 2070.0
    assert w["power_w_max"] == 1000.0
    assert w["reasons"] == ["sw_power_cap"]  # the slowdown outside the windows is not counted
    assert w["sm_max_mhz"] == 2070.0


def test_clock_window_without_nvidia_smi():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    s.rows = []
    w = s.window([(0.0, 1.0)])
    assert w["samples_under_load"] == 0 and w["sm_mhz"] is None


def test_roofline_peaks_per_bound():
    props = types.SimpleNamespace(multi_processor_count=152)
    peaks = {"bf16_tflops": 1919.0, "hbm_gbs": 6780.0}
    leg = types.SimpleNamespace(bound="tensor")
    m, spec, unit = bench.peak_of(leg, peaks, props, 2070.0)
    assert (m, unit) == (1919.0, "TFLOP/s") and abs(spec - 2577.53088) < 1e-6
    leg.bound = "tensor_tf32"
    m, spec, _ = bench.peak_of(leg, peaks, props, 2070.0)
    assert abs(m - 1919.0 * 1.1 / 2.25) < 1e-9 and abs(spec - 2577.53088 / 2) < 1e-6
    leg.bound = "hbm"
    assert bench.peak_of(leg, peaks, props, 2070.0) == (6780.0, 8000.0, "GB/s")
    leg.bound = "alu"
    m, spec, _ = bench.peak_of(leg, peaks, props, 2070.0)
    assert abs(m - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-9 and m == spec
