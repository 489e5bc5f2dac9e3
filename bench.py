#!/usr/bin/env python
"""Benchmark: fp64 PCG iterations/s and achieved HBM GB/s on the
1024 x 1024 x 128 graded, variable-coefficient anisotropic workload.

One step = one pass of the whole hot path on one right-hand side: the
per-operator set-up (level tables, face values, per-cell diagonal and Thomas
factors), the initial residual, the interleaved PCG loop to a 1e-10 relative
residual (preconditioner sweep + SpMV sweep per iteration, reductions on the
device) and the deferred solution update.  Inputs are resident in HBM before
the timed region; every vector (1.07 GB) is larger than the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With --impl reference the CPU oracle (plain
sequential C, 1 thread) is timed instead, on a bounded sample of the same
workload: a fixed number of PCG iterations on the full grid per step.
Under torchrun (N > 1) every rank solves its own copy of the workload
(replicas, weak scaling); the path has no collective.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "PCG iters/s & achieved HBM GB/s (fp64, 1024x1024x128 grid) vs HBM roofline"
UNIT = "iters/s"
# fp64 pipe operations per cell (FMA, MUL and ADD each count one) of the two
# sweeps in this implementation; see the kernel sources.
# The stencil sweep's entries are keyed by (layout, "a_h varies per column",
# form of A z).  "stencil": the full 7-point stencil (the row-tiled sweep of an
# a_h field reads per-cell horizontal weights: 4 FMAs instead of 5
# operations).  "residual": A z = r + (A - M) z, the four horizontal terms
# alone (the column layout weights its face values: one product more).
OPS_SPMV = {("tiled", True, "stencil"): 11, ("tiled", False, "stencil"): 11,
            ("column", True, "stencil"): 12, ("column", False, "stencil"): 11,
            ("tiled", True, "residual"): 8, ("tiled", False, "residual"): 8,
            ("column", True, "residual"): 9, ("column", False, "residual"): 8}
OPS_PRECOND = 6
# Algorithmic bytes per cell: vectors read/written once per sweep.
# u,p,z,q (+ per-cell diagonal, + 2 per-cell weights in the row-tiled layout)
# read, or u,p,z,q,r (+ 2 weights) for the residual form; u,p,q written
BYTES_SPMV = {("tiled", True, "stencil"): 80, ("tiled", False, "stencil"): 56,
              ("column", True, "stencil"): 64, ("column", False, "stencil"): 56,
              ("tiled", True, "residual"): 80, ("tiled", False, "residual"): 64,
              ("column", True, "residual"): 64, ("column", False, "residual"): 64}
BYTES_PRECOND = {True: 48, False: 32}  # r,q (+ 2 per-cell Thomas factors) read; r,z written
# With the factors of an a_h field rebuilt in every sweep (--factors recompute):
# the stencil sweep forms the four horizontal weights (and, in the stencil
# form, the diagonal: a product and a sum), the preconditioner sweep the
# diagonal, the pivot and the two quotients (the reciprocal and the division
# counted as one operation each: a lower bound), and neither reads per-cell
# coefficients.
OPS_BYTES_SPMV_RECOMPUTE = {"stencil": (17, 56), "residual": (12, 64)}
OPS_PRECOND_RECOMPUTE, BYTES_PRECOND_RECOMPUTE = 12, 32
# Multigrid V-cycle (--preconditioner multigrid), per cell of the level a
# kernel runs on: fp64 operations and algorithmic bytes with an a_h field
# (constant a_h: no per-cell diagonal, weights or factors), from the kernel
# sources.  first: x = omega M^-1 b (finest level: also r -= alpha q and
# ||r||^2); smooth: residual
# stencil, Thomas, x + omega z (finest level's last step: also <r, z>);
# restrict: the fine residual and 3 adds per 4 fine cells, per fine cell;
# prolong: one add per fine cell.
# restrict after one smoothing step from zero (nu = 1) takes the residual from
# the horizontal terms alone: 5 operations and 3 adds per 4 fine cells.
MG_OPS = {"first_fused": 6, "first": 4, "smooth": 12, "smooth_fused": 13, "restrict": 8.75,
          "restrict_first": 5.75, "prolong": 1}
MG_BYTES = {True: {"first_fused": 48, "first": 32, "smooth": 64, "smooth_fused": 64,
                   "restrict": 42, "restrict_first": 34, "prolong": 18},
            False: {"first_fused": 32, "first": 16, "smooth": 24, "smooth_fused": 24,
                    "restrict": 18, "restrict_first": 18, "prolong": 18}}


def mg_vcycle_cost(nx, ny, nz, levels, nu, varying):
    """(fp64 ops, algorithmic bytes) of one V-cycle per cell of the finest grid."""
    n0 = nx * ny * nz
    ops = byt = 0.0
    for l in range(levels):
        cells = (nx >> l) * (ny >> l) * nz / n0
        ks = ["first_fused" if l == 0 else "first"] + ["smooth"] * (nu - 1)
        if l + 1 < levels:
            ks += ["restrict_first" if nu == 1 else "restrict", "prolong"] + ["smooth"] * (nu - 1)
            ks.append("smooth_fused" if l == 0 else "smooth")
        ops += cells * sum(MG_OPS[k] for k in ks)
        byt += cells * sum(MG_BYTES[varying][k] for k in ks)
    return ops, byt


L2_BYTES = 129e6                     # GB300 L2
NOMINAL_HBM_GBS = 8000.0             # the ~8 TB/s HBM3e figure the fraction is also quoted on
TIMING_EVERY = 4                     # per-kernel timing in every 4th timed step
FUSED_MIN_BYTES = 88                 # u, p, z, q read + u, p, q written; r, q read + r, z written
FP64_LANES_PER_SM_CLK = 2.0          # GB300 nominal non-tensor fp64 rate: 2 FMA lanes per SM per clock
# Algorithmic bytes per cell of the paper's fused kernels (Appendix A,
# Algorithms 2 and 3) with no per-cell coefficients: the SpMV sweep reads
# u, p, z, q and writes u, p, q; the preconditioner sweep reads r, q and
# writes r, z (together FUSED_MIN_BYTES)
FUSED_MIN_BYTES_SPMV, FUSED_MIN_BYTES_PRECOND = 56, 32


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-iters", type=int, default=None,
                    help="PCG iterations of one oracle sample (default: 4 for cpu_baseline, "
                         "2 per step for --impl reference)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-standalone", action="store_true",
                    help="skip timing the standalone apply_A and precond")
    ap.add_argument("--layout", choices=["column", "tiled"], default="tiled",
                    help="layout of the solver's internal vectors")
    ap.add_argument("--factors", choices=["stored", "recompute"], default="stored",
                    help="per-cell factors of an a_h field read from arrays or rebuilt in "
                         "every sweep (row-tiled layout)")
    ap.add_argument("--substructuring", type=int, default=0,
                    help="blocks per column of the substructured preconditioner solve "
                         "(0 automatic, 1 off, 2/4/8/16)")
    ap.add_argument("--az-form", choices=["auto", "stencil", "residual"], default="auto",
                    help="how the stencil sweep forms A z: the full 7-point stencil, or "
                         "r + (A - M) z from the preconditioner sweep's M z = r")
    ap.add_argument("--preconditioner", choices=["line", "multigrid"], default="line",
                    help="column (line) solve of eq. (19), or one V-cycle of tensor-product "
                         "multigrid with it as smoother")
    ap.add_argument("--mg-levels", type=int, default=0,
                    help="multigrid levels at most (0: coarsen while nx and ny are even)")
    ap.add_argument("--loop", choices=["auto", "batched", "persistent", "cluster"],
                    default="auto", help="solve loop (row-tiled layout)")
    ap.add_argument("--grid", type=int, nargs=3, metavar=("NX", "NY", "NZ"),
                    help="same coefficients on another grid size (profiling captures)")
    ap.add_argument("--cpu-all", action="store_true",
                    help="time the CPU oracle (1 thread) on every workload with its own "
                         "stopping rule, one JSON line per workload (no GPU work)")
    ap.add_argument("--cpu-openmp", action="store_true",
                    help="with --cpu-all: the same oracle source built with -fopenmp, on every "
                         "host thread")
    ap.add_argument("--no-cpu-openmp", action="store_true",
                    help="leave out the cpu_baseline_openmp line")
    ap.add_argument("--cpu-omp-sample", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self._summary = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Median SM clock, maximum and active throttle reasons; read once
        from the sample file, then cached."""
        if self._summary is not None:
            return self._summary
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        self._summary = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                         "reasons": sorted(reasons), "samples": len(sm)}
        return self._summary


def reduce_over_ranks(ms, iters, device):
    """(max over ranks of the timed milliseconds, sum over ranks of the
    iterations).  Every rank solves its own copy of the workload (replicas),
    so the job's throughput is the summed work over the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(iters)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    n = torch.tensor([float(iters)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def host_cpu():
    """(logical CPUs, CPU model name) of the host the oracle runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return os.cpu_count(), model


def fp64_probe():
    """The library's fp64-rate probe (8 independent FMA chains per thread, the
    fastest of 3 launches of about 20 ms): one warp per SM, whose
    sub-partition's pipe it measures alone, and 32 warps per SM, all four
    sub-partitions streaming back-to-back fp64 work."""
    import matrix_free_pcg_gb300 as mf
    one = mf.pcg_measure_fp64_rate(1, 3)
    allsp = mf.pcg_measure_fp64_rate(32, 3)
    return {"per_subpartition": one, "all_subpartitions": allsp,
            "lanes_per_sm_clk": 4.0 * one["lanes_per_sm_clk"]}


def sources_sha256(names):
    """sha256 over the code of the named kernel sources (csrc/), concatenated in
    order, with comments and whitespace removed: a capture stays valid across
    comment edits and goes stale with any change of the code itself."""
    import hashlib
    import re
    hsh = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "matrix_free_pcg_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        hsh.update(" ".join(text.split()).encode())
    return hsh.hexdigest()


def measured_traffic(kernel, cells, layout, factors, az_form):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when no capture matches the layout, the
    factor mode, the form of A z and the size, or the kernel sources changed
    since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        for c in t["captures"]:
            if ((c["layout"], c["factors"], c.get("az_form", "stencil"), c["full_cells"])
                    != (layout, factors, az_form, cells)):
                continue
            if c["sha256"] != sources_sha256(c["sources"]) or kernel not in c["kernels"]:
                return None
            return c["kernels"][kernel]["bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None
    return None


def workload_inputs(w):
    """(h, a_h field, vector): the right-hand side, or for a manufactured
    workload the solution u* whose image b = A u* the caller forms."""
    return W.make_inputs(w)


def oracle_rhs(w, h, ah, vec):
    """b on the host for the oracle legs (b = A u* by the oracle's own operator
    for a manufactured workload)."""
    if w.rhs != "manufactured":
        return vec
    import oracle
    prob = oracle.Problem(w.nx, w.ny, w.nz, ah=ah, a_v=w.a_v, mass=w.mass, h=h)
    return oracle.apply_A(prob, vec)


def cpu_oracle_sample(w, h, ah, b, iters, multigrid=False):
    """The oracle as it stands on the full grid, `iters` fixed iterations
    (with the multigrid preconditioner: the oracle's MG-PCG)."""
    import oracle
    prob = oracle.Problem(w.nx, w.ny, w.nz, ah=ah, a_v=w.a_v, mass=w.mass, h=h)
    t0 = time.perf_counter()
    solve = oracle.mg_pcg if multigrid else oracle.pcg
    _, it, _, _ = solve(prob, b, rtol=0.0, maxit=iters)
    dt = time.perf_counter() - t0
    return it, dt


def openmp_threads():
    """Threads the OpenMP build of the oracle uses in this process (its
    runtime is loaded with the library)."""
    import ctypes
    try:
        return int(ctypes.CDLL("libgomp.so.1").omp_get_max_threads())
    except (OSError, AttributeError):
        return None


def run_cpu_omp_sample(args, w):
    """Child process of cpu_openmp_sample: the OpenMP build (ORACLE_LIB) on the
    full grid, args.cpu_iters fixed iterations; one JSON line."""
    h, ah, vec = workload_inputs(w)
    b = oracle_rhs(w, h, ah, vec)
    it, dt = cpu_oracle_sample(w, h, ah, b, args.cpu_iters)
    print(json.dumps({"iters": it, "seconds": dt, "threads": openmp_threads()}), flush=True)
    return 0


def cpu_openmp_sample(args, w, iters):
    """The same oracle source built with -fopenmp (loops over cells and columns
    on every host thread, dot products in per-thread parts), timed like the
    sequential sample in a child process on the same workload.  Returns the
    cpu_baseline_openmp object, or one that says why there is none."""
    try:
        from oracle import build as obuild
        lib = obuild.build(openmp=True)
    except (OSError, subprocess.SubprocessError) as e:
        return {"unavailable": "the OpenMP build of the oracle failed: %s" % e}
    ncpu, model = host_cpu()
    env = dict(os.environ, ORACLE_LIB=lib)
    env.setdefault("OMP_NUM_THREADS", str(ncpu))
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-omp-sample", "--workload",
           args.workload, "--cpu-iters", str(iters)]
    if args.grid:
        cmd += ["--grid"] + [str(v) for v in args.grid]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900,
                             check=True).stdout
        res = json.loads(out.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"unavailable": "the OpenMP sample failed: %s" % e}
    return {"value": res["iters"] / res["seconds"], "unit": UNIT, "cores": res["threads"],
            "kind": "oracle_openmp", "host_cpus": ncpu, "cpu_model": model,
            "sample": "oracle_pcg built with -fopenmp from the same source (cells and columns "
                      "on every thread, per-thread partial dot products), the full %dx%dx%d "
                      "grid, %d fixed PCG iterations (initial residual and first preconditioner "
                      "solve included), %s threads of %d (%s), %.1f s"
                      % (w.nx, w.ny, w.nz, res["iters"], res["threads"], ncpu, model,
                         res["seconds"])}


def run_reference(args, w):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    h, ah, vec = workload_inputs(w)
    b = oracle_rhs(w, h, ah, vec)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, h, ah, b, args.cpu_iters)
    tot_it, tot_t = 0, 0.0
    for _ in range(args.steps):
        it, dt = cpu_oracle_sample(w, h, ah, b, args.cpu_iters)
        tot_it += it
        tot_t += dt
    value = tot_it / tot_t
    ncpu, model = host_cpu()
    sample = ("oracle_pcg on the full %dx%dx%d grid, %d fixed PCG iterations per step "
              "(initial residual and first preconditioner solve included), sequential C, "
              "1 thread of %d (%s)" % (w.nx, w.ny, w.nz, args.cpu_iters, ncpu, model))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "grid": [w.nx, w.ny, w.nz], "iters_per_step":
                   args.cpu_iters, "l2": "inputs larger than L2"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "host_cpus": ncpu, "cpu_model": model, "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_cpu_all(args):
    """The oracle as it stands, sequential C on 1 host thread, on all five
    workloads with their own stopping rules (the CPU rows of the paper's
    section 7 Tables 5 and 6): iterations, time to solution, iterations/s and
    the bandwidth those iterations imply at the fused minimum of 88 B/cell."""
    rank, _, _ = rank_info()
    if rank != 0:
        return 0
    ncpu, model = host_cpu()
    if args.cpu_openmp:
        from oracle import build as obuild
        os.environ["ORACLE_LIB"] = obuild.build(openmp=True)
        os.environ.setdefault("OMP_NUM_THREADS", str(ncpu))
    import oracle
    threads = (openmp_threads() if args.cpu_openmp else 1)
    for name in sorted(W.WORKLOADS, key=lambda k: W.WORKLOADS[k].n):
        w = W.WORKLOADS[name]
        h, ah, vec = workload_inputs(w)
        b = oracle_rhs(w, h, ah, vec)
        prob = oracle.Problem(w.nx, w.ny, w.nz, ah=ah, a_v=w.a_v, mass=w.mass, h=h)
        t0 = time.perf_counter()
        _, it, hist, st = oracle.pcg(prob, b, rtol=w.rtol, maxit=w.maxit)
        dt = time.perf_counter() - t0
        print(json.dumps({
            "impl": "oracle_openmp" if args.cpu_openmp else "oracle", "workload": name,
            "grid": [w.nx, w.ny, w.nz], "cells": w.n,
            "rtol": w.rtol, "maxit": w.maxit, "iters": it, "status": st,
            "final_rel_residual": float(hist[-1]), "time_to_solution_s": dt,
            "iters_per_s": it / dt, "fused_min_gbs": FUSED_MIN_BYTES * w.n * it / dt / 1e9,
            "cores": threads, "host_cpus": ncpu, "cpu_model": model,
            "what": "oracle_pcg from x0 = 0: initial residual, every iteration and the "
                    "final update; " + ("the same source built with -fopenmp"
                                        if args.cpu_openmp else
                                        "sequential C, -O2 -ffp-contract=off")}), flush=True)
    return 0


def run_ours(args, w):
    import torch
    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import matrix_free_pcg_gb300 as mf

    h, ah, vec = workload_inputs(w)
    varying = w.varying_ah
    coeffs = dict(a_h=w.a_h, a_h_field=ah if varying else None, a_v=w.a_v, mass=w.mass, dz=h)
    solver = mf.Solver(w.nx, w.ny, w.nz, **coeffs)
    stream = torch.cuda.current_stream(dev)
    solver.set_stream(stream)
    bd = torch.from_numpy(vec).to(dev)
    if w.rhs == "manufactured":  # b = A u*, formed by the library's own operator
        bd = solver.apply_A(bd)
    b = bd.cpu().numpy()
    x = torch.zeros_like(bd)
    solver.set_layout(args.layout)
    solver.set_factors(args.factors)
    solver.set_substructuring(args.substructuring)
    solver.set_az_form(args.az_form)
    solver.set_loop(args.loop)
    mgrid = args.preconditioner == "multigrid"
    if mgrid:
        solver.set_multigrid(1, 0.8, args.mg_levels)
        solver.set_preconditioner("multigrid")
    az_form = solver.az_form
    recompute = args.factors == "recompute" and varying and args.layout == "tiled"

    def step():
        solver.update_coeffs(**coeffs)
        # from x0 = 0: the library neither reads x nor needs it filled
        it, _, st = solver.solve_from_zero(bd, x, rtol=w.rtol, maxit=w.maxit, history=False)
        if st not in (mf.PCG_OK,):
            raise RuntimeError("solve status %d: %s" % (st, mf.pcg_last_error(solver.ctx)))
        return it

    # warm-up; its first step with per-kernel timing, so that the library holds
    # its CUDA graphs both with and without timing events before the timed steps
    for i in range(max(args.warmup, 3)):
        solver.enable_timing(i == 0)
        step()
    solver.enable_timing(False)
    probe = fp64_probe()  # the measured fp64 rate, taken before the timed steps

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    iters = []
    launches = 0
    # per-kernel timing (CUDA events between the kernels, about 0.35% of a step)
    # in every TIMING_EVERY-th timed step; the kernel times are their sums
    ktot = {}
    timed_steps, timed_iters = 0, 0
    # face values; diagonal and Thomas factors (+ substructuring tables)
    setup_launches = (2 if varying else 0) + (2 if solver.substructuring > 1 else 0)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            timed = i % TIMING_EVERY == 0
            if timed:
                solver.enable_timing(True)  # zeroes the library's counters
            iters.append(step())
            launches += solver.launch_info()["last_solve_launches"] + setup_launches
            if timed:
                for k, (kms, kn) in solver.kernel_times().items():
                    acc = ktot.setdefault(k, [0.0, 0])
                    acc[0] += kms
                    acc[1] += kn
                solver.enable_timing(False)
                timed_steps += 1
                timed_iters += iters[-1]
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = e0.elapsed_time(e1)
    ktimes = {k: (v[0], v[1]) for k, v in ktot.items()}
    ms_max, total_iters = reduce_over_ranks(ms, sum(iters), dev)
    value = total_iters / (ms_max * 1e-3)

    # standalone operator and preconditioner (after the timed steps; not in
    # `value`): y = A x and z = M^{-1} r on the caller's column-contiguous vectors
    standalone = None
    if not args.no_standalone:
        y = torch.empty_like(bd)
        reps = 5
        out = {}
        for name, fn in (("apply_A", lambda: solver.apply_A(bd, y)),
                         ("precond", lambda: solver.precond(bd, y))):
            fn()
            torch.cuda.synchronize()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(reps):
                fn()
            s1.record(stream)
            torch.cuda.synchronize()
            out[name] = s0.elapsed_time(s1) / reps
        # fp64 operations and algorithmic bytes per cell: the stencil 8 (field:
        # 4 horizontal, diagonal, 2 vertical, weight) or 7 (constant: 3 adds +
        # 4), x and y (+ diagonal); the Thomas solve 3 (forward 2, back 1), r
        # and z (+ 2 factors)
        ops = {"apply_A": 8 if varying else 7, "precond": 3}
        byt = {"apply_A": 24 if varying else 16, "precond": 32 if varying else 16}
        clk_s = clocks.summary() or {}
        nsm_s = torch.cuda.get_device_properties(dev).multi_processor_count
        peak_s = probe["lanes_per_sm_clk"] * nsm_s * (clk_s.get("sm_mhz") or
                                                       probe["per_subpartition"]["sm_mhz"]) / 1e3
        standalone = {k: {"ms": v, "fp64_gops": ops[k] * w.n / (v * 1e-3) / 1e9,
                          "frac_fp64": ops[k] * w.n / (v * 1e-3) / 1e9 / peak_s,
                          "gbs": byt[k] * w.n / (v * 1e-3) / 1e9,
                          "ops_per_cell": ops[k], "bytes_per_cell": byt[k]}
                      for k, v in out.items()}
        del y

    n = w.n
    peaks, peak_src = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    clk = clocks.summary()
    key = (args.layout, varying, az_form)
    ops_a, bytes_a = (OPS_BYTES_SPMV_RECOMPUTE[az_form] if recompute
                      else (OPS_SPMV[key], BYTES_SPMV[key]))
    ops_m, bytes_m = ((OPS_PRECOND_RECOMPUTE, BYTES_PRECOND_RECOMPUTE) if recompute
                      else (OPS_PRECOND, BYTES_PRECOND[varying]))
    if mgrid:  # the preconditioner step is one V-cycle (the stored factors)
        key = (args.layout, varying, "stencil")
        ops_a, bytes_a = OPS_SPMV[key], BYTES_SPMV[key]
        ops_m, bytes_m = mg_vcycle_cost(w.nx, w.ny, w.nz, solver.multigrid_levels, 1, varying)
    bytes_iter = (bytes_a + bytes_m) * n
    ops_iter = (ops_a + ops_m) * n
    # the first iteration of a batched row-tiled solve runs the first-iteration
    # sweeps (alpha = beta = 0, p = q = 0 not read): 3 + 1 fp64 operations and
    # 32 + 16 bytes per cell fewer than a full iteration, once per solve
    per_solve = lambda k: ktimes.get(k, (0.0, 0))[1] / max(timed_steps, 1)  # noqa: E731
    saved_ops = (3 * per_solve("spmv_first") + per_solve("precond_first")) * n
    saved_bytes = (32 * per_solve("spmv_first") + 16 * per_solve("precond_first")) * n
    hbm_gbs = ((bytes_iter * (total_iters / world) - saved_bytes * args.steps)
               / (ms_max * 1e-3) / 1e9)

    # roofline of the dominant kernel, from its live CUDA-event times; a
    # persistent loop (small grids) is one kernel for all iterations of a solve
    kinds = {"spmv_fused": (ops_a, bytes_a), "precond_fused": (ops_m, bytes_m),
             "loop": (ops_a + ops_m, bytes_a + bytes_m)}
    dom = max(kinds, key=lambda k: ktimes[k][0])
    dom_ms, dom_n = ktimes[dom]
    if dom == "loop":  # per iteration: the loop's time over the iterations it ran
        dom_n = max(timed_iters, 1)
    avg_s = dom_ms * 1e-3 / max(dom_n, 1)
    ops_cell, bytes_cell = kinds[dom]
    sm_mhz = (clk or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    # the measured fp64 rate: the probe's lane operations per SM per clock at
    # the SM clock sampled during the timed steps (G fp64 ops / s)
    alu_peak = probe["lanes_per_sm_clk"] * nsm * sm_mhz / 1e3
    alu_nominal = FP64_LANES_PER_SM_CLK * nsm * sm_mhz * 1e6 / 1e9
    alu_ach = ops_cell * n / avg_s / 1e9
    hbm_ach = bytes_cell * n / avg_s / 1e9
    traffic = measured_traffic(dom, n, args.layout, args.factors, az_form)
    # the same launch against HBM with the algorithmic bytes of the paper's
    # fused kernels without per-cell coefficients
    fused_cell = {"spmv_fused": FUSED_MIN_BYTES_SPMV, "precond_fused": FUSED_MIN_BYTES_PRECOND,
                  "loop": FUSED_MIN_BYTES}[dom]
    roofline = {
        "bound": "alu", "kernel": "mg_vcycle" if (mgrid and dom == "precond_fused") else dom,
        "achieved": alu_ach, "peak": alu_peak,
        "unit": "G fp64 ops/s", "frac": alu_ach / alu_peak, "traffic": traffic,
        "peak_source": ("measured: fp64-rate probe, one warp per SM retires %.3f lanes/clk on its "
                        "sub-partition (8 independent FMA chains per thread, %.0f MHz inside the "
                        "probe) x 4 sub-partitions x %d SMs x %.0f MHz (median under load); with "
                        "all four sub-partitions streaming back-to-back FMAs the probe caps at "
                        "%.3f lanes/SM/clk"
                        % (probe["per_subpartition"]["lanes_per_sm_clk"],
                           probe["per_subpartition"]["sm_mhz"], nsm, sm_mhz,
                           probe["all_subpartitions"]["lanes_per_sm_clk"])),
        "peak_nominal": alu_nominal, "frac_nominal": alu_ach / alu_nominal,
        "peak_nominal_source": "%.0f fp64 lanes/SM/clk x %d SMs x %.0f MHz"
                               % (FP64_LANES_PER_SM_CLK, nsm, sm_mhz),
        "fp64_probe": probe,
        "ops_per_cell": ops_cell, "bytes_per_cell": bytes_cell,
        "avg_launch_ms": avg_s * 1e3, "launches": dom_n,
        "hbm_achieved_gbs": hbm_ach, "hbm_peak_gbs": hbm_peak,
        "hbm_frac": hbm_ach / hbm_peak, "hbm_peak_source": peak_src,
        "hbm_fused_min": {"bytes_per_cell": fused_cell,
                       "achieved_gbs": fused_cell * n / avg_s / 1e9,
                       "frac": fused_cell * n / avg_s / 1e9 / hbm_peak},
    }
    kernels = {k: {"ms": v[0], "launches": v[1], "ms_per_launch": v[0] / v[1],
                   "timed_steps": timed_steps, "of_steps": args.steps}
               for k, v in ktimes.items() if v[1]}
    # the iteration loop alone (both sweeps, or the persistent loop), per
    # solve, and the bandwidth it implies at the fused minimum of 88 B/cell
    # per iteration (u, p, z, q, r moved once, no per-cell coefficients)
    loop_ms = (sum(ktimes.get(k, (0.0, 0))[0] for k in ("precond_fused", "spmv_fused", "loop",
                                                        "precond_first", "spmv_first"))
               / max(timed_steps, 1))
    iters_solve = timed_iters / max(timed_steps, 1)
    loop_stats = {
        "ms_per_solve": loop_ms, "iters_per_solve": iters_solve,
        "ms_per_iter": loop_ms / max(iters_solve, 1),
        "algorithmic_gbs": ((bytes_iter * iters_solve - saved_bytes)
                            / (loop_ms * 1e-3) / 1e9),
        "fused_min_gbs": FUSED_MIN_BYTES * n * iters_solve / (loop_ms * 1e-3) / 1e9,
    }
    loop_stats["algorithmic_frac"] = loop_stats["algorithmic_gbs"] / hbm_peak
    loop_stats["fused_min_frac"] = loop_stats["fused_min_gbs"] / hbm_peak
    loop_stats["fused_min_frac_nominal_8tbs"] = loop_stats["fused_min_gbs"] / NOMINAL_HBM_GBS
    loop_stats["fp64_gops"] = (ops_iter * iters_solve - saved_ops) / (loop_ms * 1e-3) / 1e9
    loop_stats["fp64_frac"] = loop_stats["fp64_gops"] / alu_peak
    # DRAM bytes of one iteration (both sweeps, from the committed ncu captures)
    # against the fused minimum of 88 B/cell (u, p, z, q, r moved once, no
    # per-cell coefficients) and against the sweeps' own algorithmic bytes (with the per-cell coefficients)
    dram_iter = None
    t_m = measured_traffic("precond_fused", n, args.layout, args.factors, az_form)
    t_a = measured_traffic("spmv_fused", n, args.layout, args.factors, az_form)
    if t_m and t_a:
        # the ncu DRAM bytes of one iteration over the loop's live time per
        # iteration: the bandwidth the fused iteration sustains in DRAM terms
        dram_gbs = (t_m + t_a) / (loop_stats["ms_per_iter"] * 1e-3) / 1e9
        dram_iter = {"bytes": t_m + t_a, "per_cell": (t_m + t_a) / n,
                     "vs_fused_min_88": (t_m + t_a) / (88.0 * n),
                     "vs_algorithmic": (t_m + t_a) / bytes_iter,
                     "gbs": dram_gbs, "frac": dram_gbs / hbm_peak,
                     "frac_nominal_8tbs": dram_gbs / NOMINAL_HBM_GBS}

    # end to end through the host-buffer entry point that takes the step's
    # coefficients and right-hand side together (pcg_update_solve_host with
    # x0 = NULL): pinned b in -- copied while the set-up kernels run -- and x
    # out; one page-locked output buffer for every step, as a caller solving
    # repeatedly would keep it
    e2e = None
    if not args.no_e2e:
        nsteps = args.steps
        bh = torch.from_numpy(b).pin_memory()
        xh = torch.zeros(n, dtype=torch.float64).pin_memory()
        solver.update_solve_host(bh, xh, rtol=w.rtol, maxit=w.maxit, history=False, x0=None,
                                 **coeffs)  # warm-up
        barrier()
        torch.cuda.synchronize()
        t_e2e = 0.0
        e2e_it = 0
        step_ms, copy_ms = [], []
        for _ in range(nsteps):
            ts = time.perf_counter()
            it, _, st = solver.update_solve_host(bh, xh, rtol=w.rtol, maxit=w.maxit,
                                                 history=False, x0=None, **coeffs)
            dt = time.perf_counter() - ts
            t_e2e += dt
            e2e_it += it
            step_ms.append(round(1e3 * dt, 3))
            # copy-only control, outside the timed total: the same bytes through
            # the same page-locked buffers, one cudaMemcpyAsync each way, no solve
            tc = time.perf_counter()
            bd.copy_(bh, non_blocking=True)
            xh.copy_(x, non_blocking=True)
            torch.cuda.synchronize()
            copy_ms.append(round(1e3 * (time.perf_counter() - tc), 3))
        torch.cuda.synchronize()
        t_e2e_ms, e2e_iters = reduce_over_ranks(1e3 * t_e2e, e2e_it, dev)
        sync = {"value": e2e_iters / (1e-3 * t_e2e_ms), "unit": UNIT,
                "api": "pcg_update_solve_host (x0 = 0)", "steps": nsteps, "step_ms": step_ms,
                "copy_only_ms": copy_ms,
                "copy_only": "after each step, outside its time: the step's b in and x out "
                             "through the same page-locked buffers, no solve"}
        # the same steps as a sequence of solves through the asynchronous call:
        # each solution's copy to the host runs behind the next step's set-up
        # and solve; the timed region ends when the last copy has landed
        barrier()
        torch.cuda.synchronize()
        a_it = 0
        a_step_ms = []
        t0 = time.perf_counter()
        for _ in range(nsteps):
            ts = time.perf_counter()
            it, _, st = solver.update_solve_host_async(bh, xh, rtol=w.rtol, maxit=w.maxit,
                                                       history=False, x0=None, **coeffs)
            a_it += it
            a_step_ms.append(round(1e3 * (time.perf_counter() - ts), 3))
        solver.host_wait()
        t_async = time.perf_counter() - t0
        t_async_ms, a_iters = reduce_over_ranks(1e3 * t_async, a_it, dev)
        e2e = {"value": a_iters / (1e-3 * t_async_ms), "unit": UNIT,
               # b, plus the coefficient arrays the step hands over (a_h field, dz)
               "h2d_bytes_per_step": 8 * n + (8 * w.nx * w.ny if varying else 0) + 8 * w.nz,
               "d2h_bytes_per_step": 8 * n,
               "api": "pcg_update_solve_host_async (x0 = 0) per step, pcg_host_wait after the "
                      "last: each step's b in and x out inside the timed region, x's copy "
                      "running behind the next step's solve",
               "steps": nsteps, "step_ms": a_step_ms, "sync": sync}
        del xh, bh

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        mgi = max(1, args.cpu_iters // 2) if mgrid else args.cpu_iters
        it_c, dt_c = cpu_oracle_sample(w, h, ah, oracle_rhs(w, h, ah, vec), mgi, mgrid)
        ncpu, model = host_cpu()
        cpu = {"value": it_c / dt_c, "unit": UNIT, "cores": 1, "kind": "oracle",
               "host_cpus": ncpu, "cpu_model": model,
               "sample": "%s on the full %dx%dx%d grid, %d fixed PCG iterations "
                         "(initial residual and first preconditioner solve included), "
                         "sequential C, 1 thread of %d (%s), %.1f s"
                         % ("oracle_mg_pcg" if mgrid else "oracle_pcg", w.nx, w.ny, w.nz, mgi,
                            ncpu, model, dt_c)}
    cpu_omp = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.no_cpu_openmp:
        cpu_omp = ({"unavailable": "the OpenMP build parallelises the line-preconditioned "
                                   "PCG only"} if mgrid else
                   cpu_openmp_sample(args, w, args.cpu_iters))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "grid": [w.nx, w.ny, w.nz], "cells": n,
                       "rtol": w.rtol, "iters_per_step": iters[0], "a_v": w.a_v,
                       "graded": w.graded, "varying_ah": varying,
                       "l2": ("inputs larger than L2 (%.2f GB per vector)" % (8e-9 * n)
                              if 8 * n > L2_BYTES else
                              "working set L2-resident (%.1f MB per vector), no flush"
                              % (8e-6 * n)),
                       "layout": args.layout, "factors": args.factors,
                       "substructuring": solver.substructuring, "az_form": az_form,
                       "loop": solver.loop,
                       "preconditioner": args.preconditioner,
                       "multigrid": ({"levels": solver.multigrid_levels, "nu": 1, "omega": 0.8}
                                     if mgrid else None),
                       "parallelism": "replicas" if world > 1 else "single"},
            "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / hbm_peak,
            "hbm_frac_nominal_8tbs": hbm_gbs / NOMINAL_HBM_GBS,
            "loop": loop_stats,
            "bytes_per_cell_iter": bytes_iter / n, "fp64_ops_per_cell_iter": ops_iter / n,
            "dram_per_iter": dram_iter, "standalone": standalone,
            "roofline": roofline, "kernels": kernels, "clocks": clk, "e2e": e2e,
            "cpu_baseline": cpu, "cpu_baseline_openmp": cpu_omp, "gpu_launches": launches,
            "time_to_solution_ms": ms_max / args.steps,
        }
        print(json.dumps(line), flush=True)
    solver.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.cpu_iters is None:
        args.cpu_iters = 2 if args.impl == "reference" else 4
    w = W.WORKLOADS[args.workload]
    if args.grid:
        import dataclasses
        nx, ny, nz = args.grid
        w = dataclasses.replace(w, name="%s_on_%dx%dx%d" % (w.name.rsplit("_", 1)[0], nx, ny, nz),
                                nx=nx, ny=ny, nz=nz)
    if args.cpu_all:
        return run_cpu_all(args)
    if args.cpu_omp_sample:
        return run_cpu_omp_sample(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
