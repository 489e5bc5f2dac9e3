"""Build libpcg.so (the CUDA kernels and the C ABI) for sm_103a, in-tree.

nvcc compiles each translation unit in its own process (in parallel) and
links them into matrix_free_pcg_gb300/_build/libpcg.so.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpcg.so")
SOURCES = ["pcg_kernels.cu", "pcg_setup.cu", "pcg_tiled.cu", "pcg_persistent.cu", "pcg_split.cu",
           "pcg_mg.cu", "pcg_cluster.cu", "pcg_api.cu", "pcg_noalloc.cu", "pcg_peak.cu",
           "pcg_tmem.cu"]
HEADERS = [os.path.join(CSRC, "pcg_internal.h"), os.path.join(CSRC, "pcg_device.cuh"),
           os.path.join(CSRC, "pcg_sweeps.cuh"), os.path.join(CSRC, "pcg_tmem.cuh"),
           os.path.join(ROOT, "include", "pcg.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code (the per-level tables) is compiled without floating-point
# contraction, so it rounds like its plain definition on every host.
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xcompiler", "-ffp-contract=off", "--expt-relaxed-constexpr"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra_flags=()):
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    objs, procs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            cmd = [nvcc] + ARCH + FLAGS + list(extra_flags) + ["-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd))
            procs.append((cmd, subprocess.Popen(cmd)))
    for cmd, p in procs:
        if p.wait() != 0:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or procs or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
