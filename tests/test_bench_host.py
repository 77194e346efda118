"""Host-side rules of bench.py that decide what a reported fraction is measured against.
No GPU."""
import bench

PEAKS = {"bf16_tflops": 1892.0, "bf16_tflops_sustained": 1684.0,
         "clocks_under_load": {"sm_mhz_median": 1425.0}}


def test_burst_peak_when_the_clock_stays_near_its_maximum():
    assert bench.headline_peak(PEAKS, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}) == (1892.0, "bf16_tflops (burst)")
    # 1980 MHz is nearer 2070 than the 1425 MHz the sustained figure was taken at
    assert bench.headline_peak(PEAKS, {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0})[0] == 1892.0


def test_sustained_peak_when_the_clock_sits_near_the_sustained_measurement():
    assert bench.headline_peak(PEAKS, {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0}) == (1684.0, "bf16_tflops_sustained")
    # the midpoint between the two clocks decides
    assert bench.headline_peak(PEAKS, {"sm_mhz": 1747.0, "sm_max_mhz": 2070.0})[0] == 1684.0
    assert bench.headline_peak(PEAKS, {"sm_mhz": 1748.0, "sm_max_mhz": 2070.0})[0] == 1892.0


def test_without_a_sustained_clock_record_or_clock_samples():
    p = {"bf16_tflops": 1892.0, "bf16_tflops_sustained": 1684.0}
    assert bench.headline_peak(p, {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0})[0] == 1892.0
    assert bench.headline_peak(p, {"sm_mhz": 1990.0, "sm_max_mhz": 2070.0})[0] == 1684.0
    assert bench.headline_peak(p, {"sm_mhz": None, "sm_max_mhz": None})[0] == 1684.0
    assert bench.headline_peak(p, {})[0] == 1684.0


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on():
    for (workload, kernel), (nbytes, digest) in bench.TRAFFIC.items():
        assert nbytes > 0
        t = bench.kernel_traffic(workload, kernel)
        assert t == (nbytes if digest == bench.kernel_source_hash(kernel) else None)
    assert bench.kernel_traffic("no_such_workload", "ffa_fwd_kernel") is None
