"""The fp64-rate probe behind the roofline's peak: it runs, measures a rate
inside the GB300's fp64 pipe limits (2 lanes per SM per clock nominal), and
repeats to within a few percent."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import matrix_free_pcg_gb300 as mf  # noqa: E402


def test_fp64_probe_measures_a_plausible_rate():
    torch.cuda.init()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    runs = [mf.pcg_measure_fp64_rate(w, 2) for w in (8, 32)]
    for r in runs:
        assert 200.0 < r["sm_mhz"] < 2200.0, r
        assert 1.0 < r["lanes_per_sm_clk"] <= 2.05, r
        rel = r["lane_ops_per_s"] / (r["lanes_per_sm_clk"] * nsm * r["sm_mhz"] * 1e6)
        assert abs(rel - 1.0) < 1e-9, r
    a, b = (r["lanes_per_sm_clk"] for r in runs)
    assert abs(a - b) <= 0.05 * max(a, b), runs
    # one warp per SM: one sub-partition's pipe, at most its nominal half lane per clock
    one = mf.pcg_measure_fp64_rate(1, 2)
    assert 0.3 < one["lanes_per_sm_clk"] <= 0.51, one
    assert one["lanes_per_sm_clk"] * 4 >= a * 0.99, (one, runs)
