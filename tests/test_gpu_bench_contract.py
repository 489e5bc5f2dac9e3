"""bench.py's own arm on the GPU: one JSON line with every key of the
contract, on small workloads (the line's numbers are checked for
consistency with each other, not for speed)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
           *extra]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["aniso_32x32x16", "manufactured_128x128x64"])
def test_bench_line_has_the_contract_keys(workload):
    d = run_bench("--workload", workload, "--cpu-iters", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["unit"] == "iters/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 3, 3)
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["scaling"] == "weak"
    assert d["config"]["workload"] == workload
    # value = iterations per second of the timed steps
    its = d["config"]["iters_per_step"]
    assert abs(d["value"] - its / (1e-3 * d["ms_per_step"])) <= 1e-6 * d["value"]
    rl = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rl, key
    assert rl["bound"] in ("hbm", "tensor", "alu") and rl["peak"] > 0
    assert abs(rl["frac"] - rl["achieved"] / rl["peak"]) <= 1e-9 * max(1.0, rl["frac"])
    assert 0.0 < rl["frac"] < 1.5
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = d["e2e"]
    n = d["config"]["cells"]
    assert e2e["unit"] == "iters/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] >= 8 * n and e2e["d2h_bytes_per_step"] == 8 * n
    assert len(e2e["step_ms"]) == 3 and len(e2e["sync"]["copy_only_ms"]) == 3
    assert e2e["sync"]["value"] > 0 and "async" in e2e["api"]
    assert rl["peak_source"].startswith("measured") and rl["fp64_probe"]["lanes_per_sm_clk"] > 0
    assert abs(rl["frac_nominal"] - rl["achieved"] / rl["peak_nominal"]) <= 1e-9
    assert cpu["host_cpus"] >= 1 and cpu["cpu_model"]
    clk = d["clocks"]
    if clk is not None:
        assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)
    assert d["gpu_launches"] > 0


def test_bench_multigrid_line():
    d = run_bench("--workload", "aniso_32x32x16", "--preconditioner", "multigrid",
                  "--mg-levels", "4", "--no-cpu-baseline", "--no-e2e", "--no-standalone")
    assert d["config"]["preconditioner"] == "multigrid" and d["value"] > 0
    assert d["roofline"]["kernel"] == "mg_vcycle" and d["gpu_launches"] > 0
