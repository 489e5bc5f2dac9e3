"""bench.py's clock sampler: the summary of the samples taken during the
timed region is read once and stays available to every later caller (the
roofline peak and the `clocks` key of the JSON line)."""
import os
import sys
import tempfile

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


class _Done:
    """Stands in for the finished nvidia-smi process."""


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = _Done()
    return s


def test_summary_is_stable_across_calls():
    s = _sampler_with([
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 910.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 905.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    first = s.summary()
    assert first == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                     "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(s.path)
    assert s.summary() == first


def test_summary_of_no_samples_is_none():
    s = _sampler_with(["garbage"])
    assert s.summary() is None
