"""The OpenMP build of the oracle (a timing baseline for the benchmark's
cpu_baseline_openmp line) against the sequential build of the same source.

Per-cell and per-column work (apply_A, the column solves) is the same
arithmetic in both builds, so it must agree bit for bit; the PCG dot products
add per-thread partial sums in the OpenMP build, so its iterates agree to
rounding and its iteration counts exactly on these well-separated cases.
Each build runs in its own process (the library is chosen when the oracle
package loads)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle
import workloads as W
out = {}
for (nx, ny, nz, vary) in [(32, 32, 16, True), (48, 40, 24, False), (64, 64, 64, True)]:
    h = W.layer_thickness(nz, True)
    ah = W.horizontal_coefficient(nx, ny, vary)
    prob = oracle.Problem(nx, ny, nz, ah=ah, a_v=10.0, mass=1.0, h=h)
    b = np.random.default_rng(3).uniform(-1, 1, nx * ny * nz)
    key = "%dx%dx%d" % (nx, ny, nz)
    np.save(sys.argv[2] + "/%s_A.npy" % key, oracle.apply_A(prob, b))
    np.save(sys.argv[2] + "/%s_M.npy" % key, oracle.precond(prob, b))
    x, it, hist, st = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
    np.save(sys.argv[2] + "/%s_x.npy" % key, x)
    out[key] = [it, st]
print(json.dumps(out))
"""


def run_build(lib, outdir, threads):
    env = dict(os.environ, ORACLE_LIB=lib, OMP_NUM_THREADS=str(threads))
    os.makedirs(outdir, exist_ok=True)
    res = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, outdir], env=env,
                         capture_output=True, text=True, timeout=600, check=True)
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_openmp_build_agrees_with_the_sequential_build(tmp_path):
    from oracle import build as obuild
    seq = obuild.build()
    try:
        omp = obuild.build(openmp=True)
    except (OSError, subprocess.CalledProcessError) as e:
        pytest.skip("no OpenMP build here: %s" % e)
    a = run_build(seq, str(tmp_path / "seq"), 1)
    b = run_build(omp, str(tmp_path / "omp"), 4)
    assert a == b  # iteration counts and statuses
    for key in a:
        for part in ("A", "M"):
            u = np.load(tmp_path / "seq" / ("%s_%s.npy" % (key, part)))
            v = np.load(tmp_path / "omp" / ("%s_%s.npy" % (key, part)))
            assert np.array_equal(u, v), (key, part)
        u = np.load(tmp_path / "seq" / ("%s_x.npy" % key))
        v = np.load(tmp_path / "omp" / ("%s_x.npy" % key))
        assert np.linalg.norm(u - v) <= 1e-12 * np.linalg.norm(u), key
