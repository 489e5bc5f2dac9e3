"""Compile the CPU oracle (test infrastructure only) into oracle/_build/.

Plain gcc, fp64, -O2 -ffp-contract=off, no vendor code.  Used by the test
suite, the smoke check and the benchmark's CPU-baseline leg.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle_pcg.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_pcg.so")
# the same source with -fopenmp: a timing baseline on all host cores only
LIB_OMP = os.path.join(OUT_DIR, "liboracle_pcg_omp.so")


def build(force: bool = False, openmp: bool = False) -> str:
    lib = LIB_OMP if openmp else LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(SRC):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra"] + (["-fopenmp"] if openmp else []) + [
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build(force="--force" in sys.argv, openmp=True))
