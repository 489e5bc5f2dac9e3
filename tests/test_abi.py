"""The C ABI library: it loads, exports every entry point include/pcg.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pcg.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_free_pcg_gb300 as mf
    return mf


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pcg_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["pcg_create", "pcg_destroy", "pcg_apply_A", "pcg_precond", "pcg_solve",
                     "pcg_solve_host", "pcg_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    assert sorted(lib.EXPORTED) == declared_functions()


def test_symbols_have_c_linkage(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    for n in declared_functions():
        assert n in exported


@pytest.mark.parametrize("dims", [(0, 4, 4), (4, -1, 4), (4, 4, 0)])
def test_create_rejects_bad_sizes(lib, dims):
    with pytest.raises(lib.PCGError) as e:
        lib.pcg_create(*dims)
    assert e.value.status == lib.PCG_EINVAL
    assert "must be >= 1" in lib.pcg_last_error()


@pytest.mark.parametrize("kw,msg", [({"mass": 0.0}, "mass"), ({"mass": float("nan")}, "mass"),
                                    ({"a_v": -1.0}, "a_v"), ({"a_h": -0.5}, "a_h"),
                                    ({"dz": [1.0, 0.0, 1.0]}, "dz[1]"),
                                    ({"a_h_field": [1.0] * 3 + [float("inf")]}, "a_h_field[3]"),
                                    ({"a_h_field": [1.0, float("nan"), 1.0, 1.0]}, "a_h_field[1]"),
                                    ({"a_h_field": [1.0, 1.0, -0.1, 1.0]}, "a_h_field[2]"),
                                    ({"a_h_field": [1.0, 1.0, 1.0, -float("inf")]},
                                     "a_h_field[3]")])
def test_create_rejects_bad_coefficients(lib, kw, msg):
    args = dict(a_h=1.0, a_v=10.0, mass=1.0)
    args.update(kw)
    with pytest.raises(lib.PCGError) as e:
        lib.pcg_create(2, 2, 3, **args)
    assert e.value.status == lib.PCG_EINVAL
    assert msg in lib.pcg_last_error()


def test_null_context_calls_fail_cleanly(lib):
    assert lib._lib.pcg_apply_A(None, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_precond(None, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_solve(None, None, None, 1e-10, 10, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_stream(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_solve_host(None, None, None, 1e-10, 10, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_solve_host_x0(None, None, None, None, 1e-10, 10, None, None) == \
        lib.PCG_EINVAL
    assert lib._lib.pcg_update_coeffs(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_update_solve_host(None, None, None, None, None, 1e-10, 10, None,
                                          None) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_layout(None, lib.PCG_LAYOUT_TILED) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_factors(None, lib.PCG_FACTORS_STORED) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_substructuring(None, 0) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_loop(None, lib.PCG_LOOP_AUTO) == lib.PCG_EINVAL
    assert lib._lib.pcg_get_substructuring(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_get_loop(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_test_barrier_absent(None, 0) == lib.PCG_EINVAL
    assert lib._lib.pcg_test_poison_work(None) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_az_form(None, lib.PCG_AZ_AUTO) == lib.PCG_EINVAL
    assert lib._lib.pcg_get_az_form(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_preconditioner(None, lib.PCG_PREC_LINE) == lib.PCG_EINVAL
    assert lib._lib.pcg_set_multigrid(None, 1, 0.8, 0) == lib.PCG_EINVAL
    assert lib._lib.pcg_get_multigrid(None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_mg_vcycle(None, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_precond_dot_noalloc(None, None, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_enable_timing(None, 1) == lib.PCG_EINVAL
    assert lib._lib.pcg_kernel_times(None, None, None) == lib.PCG_EINVAL
    assert lib._lib.pcg_launch_info(None, None, None, None) == lib.PCG_EINVAL
    lib._lib.pcg_destroy(None)  # NULL-safe
    assert isinstance(lib.pcg_last_error(None), str)


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(lib.PCGError) as e:
        lib.pcg_create(4, 4, 4, a_h=1.0, a_v=10.0)
    assert e.value.status == lib.PCG_ECUDA
    assert "no usable CUDA device" in lib.pcg_last_error()


def header_constants():
    """NAME = value pairs of the header's enums (comments removed)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(PCG_\w+)\s*=\s*(\d+)", text)}


def test_binding_constants_match_the_header(lib):
    consts = header_constants()
    for name, value in consts.items():
        if name.startswith("PCG_K_"):
            continue
        assert getattr(lib, name) == value, name
    # kernel kinds: the binding's list is indexed by the header's enum
    kinds = sorted((v, k) for k, v in consts.items() if k.startswith("PCG_K_") and k != "PCG_K_COUNT")
    assert len(lib.KERNEL_KINDS) == consts["PCG_K_COUNT"] == len(kinds)
    expect = {"PCG_K_PRECOND_FUSED": "precond_fused", "PCG_K_SPMV_FUSED": "spmv_fused",
              "PCG_K_RESIDUAL": "residual", "PCG_K_FINALIZE": "finalize",
              "PCG_K_APPLY_A": "apply_A", "PCG_K_PRECOND": "precond", "PCG_K_SETUP": "setup",
              "PCG_K_LOOP": "loop", "PCG_K_PRECOND_FIRST": "precond_first",
              "PCG_K_SPMV_FIRST": "spmv_first"}
    for v, k in kinds:
        assert lib.KERNEL_KINDS[v] == expect[k], (k, v)


@pytest.mark.parametrize("warps,launches", [(0, 3), (6, 3), (68, 3), (32, 0), (32, 101)])
def test_fp64_probe_rejects_bad_arguments(lib, warps, launches):
    with pytest.raises(lib.PCGError) as e:
        lib.pcg_measure_fp64_rate(warps, launches)
    assert e.value.status == lib.PCG_EINVAL
