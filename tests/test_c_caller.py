"""The C ABI from a plain C99 program (tests/c/pcg_c_caller.c): it includes
only include/pcg.h and links libpcg.so, with no Python, torch or CUDA runtime
of its own between it and the library.

On the CPU the program must compile against the header, link, and report
PCG_ECUDA from pcg_create without a GPU.  On the GPU its two solves (host
buffers in and out; then new coefficients in the one-call form) must match
the CPU oracle's: iteration counts within one, solutions within 1e-8.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "pcg_c_caller.c")
LIBDIR = os.path.join(ROOT, "matrix_free_pcg_gb300", "_build")
PCG_ECUDA = 3


def build_program(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    if not os.path.exists(os.path.join(LIBDIR, "libpcg.so")):
        pytest.skip("libpcg.so is not built")
    exe = str(tmp_path / "pcg_c_caller")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
                    "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
                    "-L", LIBDIR, "-lpcg", "-Wl,-rpath," + LIBDIR], check=True)
    return exe


def write_input(path, nx, ny, nz, a_v, mass, ah, dz, b, scale):
    with open(path, "wb") as f:
        np.array([nx, ny, nz], dtype=np.int32).tofile(f)
        np.array([a_v, mass], dtype=np.float64).tofile(f)
        np.ascontiguousarray(ah, dtype=np.float64).tofile(f)
        np.ascontiguousarray(dz, dtype=np.float64).tofile(f)
        np.ascontiguousarray(b, dtype=np.float64).tofile(f)
        np.array([scale], dtype=np.float64).tofile(f)


def case():
    nx, ny, nz, a_v, mass, scale = 37, 29, 24, 1e3, 1.0, 1.7
    dz = W.layer_thickness(nz, True)
    ah = W.horizontal_coefficient(nx, ny, True)
    b = np.random.default_rng(23).uniform(-1.0, 1.0, nx * ny * nz)
    return nx, ny, nz, a_v, mass, ah, dz, b, scale


def test_c_program_builds_and_reports_no_device(tmp_path):
    exe = build_program(tmp_path)
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the GPU test runs the program")
    nx, ny, nz, a_v, mass, ah, dz, b, scale = case()
    inp = str(tmp_path / "in.bin")
    write_input(inp, nx, ny, nz, a_v, mass, ah, dz, b, scale)
    r = subprocess.run([exe, inp, str(tmp_path / "out.bin")], capture_output=True, text=True)
    assert r.returncode == 10 + PCG_ECUDA, (r.returncode, r.stderr)
    assert "pcg_create" in r.stderr


@pytest.mark.gpu
def test_c_program_solves_like_the_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = build_program(tmp_path)
    nx, ny, nz, a_v, mass, ah, dz, b, scale = case()
    n = nx * ny * nz
    inp, outp = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    write_input(inp, nx, ny, nz, a_v, mass, ah, dz, b, scale)
    r = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stderr)
    raw = open(outp, "rb").read()
    off = 0
    results = []
    for _ in range(2):
        it, st = np.frombuffer(raw, dtype=np.int32, count=2, offset=off)
        off += 8
        x = np.frombuffer(raw, dtype=np.float64, count=n, offset=off)
        off += 8 * n
        results.append((int(it), int(st), x))
    for (it, st, x), field in zip(results, [ah, ah * scale]):
        prob = oracle.Problem(nx, ny, nz, ah=field, a_v=a_v, mass=mass, h=dz)
        x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=500)
        assert st == 0 and st_ref == oracle.OK and abs(it - it_ref) <= 1, (it, it_ref)
        assert np.linalg.norm(x - x_ref) <= 1e-8 * np.linalg.norm(x_ref)
