"""CPU oracle for the matrix-free PCG solver -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper around ``oracle_pcg.c`` (plain sequential fp64 C).
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product library never does.

Arrays use the column-contiguous layout of Mueller et al., "Matrix-free GPU
implementation of a preconditioned conjugate gradient solver for anisotropic
elliptic PDEs", section 3 eq. (10): numpy shape (ny, nx, nz), C order, so the
linear index of cell (i, j, k) is ((j*nx)+i)*nz + k.
"""
import ctypes
import os

import numpy as np

from . import build as _build

OK, EINVAL, ENOMEM, ENOTCONV, EBREAKDOWN = 0, 1, 2, 4, 5

_lib = None
_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB selects another build: a mutation test's deliberately
        # broken copy, or the benchmark's OpenMP build (oracle/build.py).
        path = os.environ.get("ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        common = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, ctypes.c_double,
                  ctypes.c_double, _dp]
        lib.oracle_apply_A.argtypes = common + [_dp, _dp]
        lib.oracle_apply_A_cells.argtypes = common + [_dp, _i64p, ctypes.c_int64, _dp]
        lib.oracle_precond.argtypes = common + [_dp, _dp]
        lib.oracle_precond_columns.argtypes = common + [_dp, _i64p, ctypes.c_int64, _dp]
        lib.oracle_pcg.argtypes = common + [_dp, _dp, ctypes.c_double, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int), _dp]
        lib.oracle_mg_levels.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_mg_level_ah.argtypes = [ctypes.c_int, ctypes.c_int, _dp, ctypes.c_int, _dp]
        lib.oracle_apply_A_area.argtypes = common + [ctypes.c_double, _dp, _dp]
        lib.oracle_mg_restrict.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp]
        lib.oracle_mg_prolong_add.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp]
        mgp = [ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_mg_vcycle.argtypes = common + mgp + [_dp, _dp]
        lib.oracle_mg_pcg.argtypes = common + mgp + [_dp, _dp, ctypes.c_double, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_int), _dp]
        for f in (lib.oracle_apply_A, lib.oracle_apply_A_cells, lib.oracle_precond,
                  lib.oracle_precond_columns, lib.oracle_pcg, lib.oracle_mg_levels,
                  lib.oracle_mg_level_ah, lib.oracle_apply_A_area, lib.oracle_mg_restrict,
                  lib.oracle_mg_prolong_add, lib.oracle_mg_vcycle, lib.oracle_mg_pcg):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s failed with oracle status %d" % (what, status))
        self.status = status


def _arr(a, n=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if n is not None and a.size != n:
        raise ValueError("expected %d values, got %d" % (n, a.size))
    return a


def _ptr(a):
    return a.ctypes.data_as(_dp)


class Problem:
    """Operator description shared by all oracle calls.

    ah: horizontal coefficient a_h(i,j) -- a scalar or an (ny, nx) array.
    a_v: vertical coefficient.  mass: zero-order coefficient.
    h: layer thicknesses (nz,), default all ones.
    """

    def __init__(self, nx, ny, nz, ah=1.0, a_v=1.0, mass=1.0, h=None):
        self.nx, self.ny, self.nz = int(nx), int(ny), int(nz)
        if np.isscalar(ah):
            ah = np.full(self.nx * self.ny, float(ah))
        self.ah = _arr(ah, self.nx * self.ny)
        self.a_v = float(a_v)
        self.mass = float(mass)
        self.h = _arr(np.ones(self.nz) if h is None else h, self.nz)

    @property
    def n(self):
        return self.nx * self.ny * self.nz

    def _common(self):
        return (self.nx, self.ny, self.nz, _ptr(self.ah), self.a_v, self.mass, _ptr(self.h))


def apply_A(prob, x):
    """y = A x (eqs. (5)-(8), (18))."""
    lib = _load()
    x = _arr(x, prob.n)
    y = np.empty(prob.n)
    st = lib.oracle_apply_A(*prob._common(), _ptr(x), _ptr(y))
    if st:
        raise OracleError(st, "oracle_apply_A")
    return y


def apply_A_cells(prob, x, cells):
    """(A x)[cells] for a list of linear cell indices."""
    lib = _load()
    x = _arr(x, prob.n)
    cells = np.ascontiguousarray(cells, dtype=np.int64)
    out = np.empty(cells.size)
    st = lib.oracle_apply_A_cells(*prob._common(), _ptr(x),
                                  cells.ctypes.data_as(_i64p), cells.size, _ptr(out))
    if st:
        raise OracleError(st, "oracle_apply_A_cells")
    return out


def precond(prob, r):
    """z = M^{-1} r, M = blockdiag of the column matrices (eq. (19))."""
    lib = _load()
    r = _arr(r, prob.n)
    z = np.empty(prob.n)
    st = lib.oracle_precond(*prob._common(), _ptr(r), _ptr(z))
    if st:
        raise OracleError(st, "oracle_precond")
    return z


def precond_columns(prob, r, cols):
    """M^{-1} r restricted to the listed columns (index j*nx+i); (len(cols), nz)."""
    lib = _load()
    r = _arr(r, prob.n)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty((cols.size, prob.nz))
    st = lib.oracle_precond_columns(*prob._common(), _ptr(r),
                                    cols.ctypes.data_as(_i64p), cols.size, _ptr(out))
    if st:
        raise OracleError(st, "oracle_precond_columns")
    return out


def pcg(prob, b, x0=None, rtol=1e-10, maxit=500, check=True):
    """Textbook PCG.  Returns (x, iters, hist, status)."""
    lib = _load()
    b = _arr(b, prob.n)
    x = np.zeros(prob.n) if x0 is None else _arr(x0, prob.n).copy()
    hist = np.full(maxit + 1, np.nan)
    iters = ctypes.c_int(-1)
    st = lib.oracle_pcg(*prob._common(), _ptr(b), _ptr(x), float(rtol), int(maxit),
                        ctypes.byref(iters), _ptr(hist))
    if check and st not in (OK, ENOTCONV):
        raise OracleError(st, "oracle_pcg")
    return x, iters.value, hist[: max(iters.value, 0) + 1], st


# ---------------------------------------------------------------- multigrid
# Tensor-product multigrid with the column solve as smoother (the paper's
# sections 1, 2 and 9; readings of the open parts in oracle_pcg.c).

MG_NU, MG_OMEGA = 1, 0.8   # defaults: one smoothing step each way, damping 0.8


def mg_levels(nx, ny, max_levels=0):
    """Number of levels of the horizontal semi-coarsening hierarchy."""
    return _load().oracle_mg_levels(int(nx), int(ny), int(max_levels))


def mg_level_ah(prob, level):
    """a_h of multigrid level `level`, shape (ny >> level, nx >> level)."""
    lib = _load()
    nxc, nyc = prob.nx >> level, prob.ny >> level
    out = np.empty(nxc * nyc)
    st = lib.oracle_mg_level_ah(prob.nx, prob.ny, _ptr(prob.ah), int(level), _ptr(out))
    if st:
        raise OracleError(st, "oracle_mg_level_ah")
    return out.reshape(nyc, nxc)


def apply_A_area(prob, x, area):
    """y = A x with the zero-order and vertical terms scaled by the
    horizontal cell area (the operator of a multigrid level)."""
    lib = _load()
    x = _arr(x, prob.n)
    y = np.empty(prob.n)
    st = lib.oracle_apply_A_area(*prob._common(), float(area), _ptr(x), _ptr(y))
    if st:
        raise OracleError(st, "oracle_apply_A_area")
    return y


def mg_restrict(nx, ny, nz, rf):
    """R rf: per layer, sums over the 2x2 fine columns of each coarse column."""
    lib = _load()
    rf = _arr(rf, nx * ny * nz)
    rc = np.empty((nx // 2) * (ny // 2) * nz)
    st = lib.oracle_mg_restrict(nx, ny, nz, _ptr(rf), _ptr(rc))
    if st:
        raise OracleError(st, "oracle_mg_restrict")
    return rc


def mg_prolong_add(nx, ny, nz, ec, xf):
    """xf + P ec (piecewise constant over the 2x2 fine columns)."""
    lib = _load()
    ec = _arr(ec, (nx // 2) * (ny // 2) * nz)
    out = _arr(xf, nx * ny * nz).copy()
    st = lib.oracle_mg_prolong_add(nx, ny, nz, _ptr(ec), _ptr(out))
    if st:
        raise OracleError(st, "oracle_mg_prolong_add")
    return out


def mg_vcycle(prob, r, nu=MG_NU, omega=MG_OMEGA, max_levels=0):
    """z = B r: one V-cycle."""
    lib = _load()
    r = _arr(r, prob.n)
    z = np.empty(prob.n)
    st = lib.oracle_mg_vcycle(*prob._common(), int(nu), float(omega), int(max_levels),
                              _ptr(r), _ptr(z))
    if st:
        raise OracleError(st, "oracle_mg_vcycle")
    return z


def mg_pcg(prob, b, x0=None, rtol=1e-10, maxit=500, nu=MG_NU, omega=MG_OMEGA, max_levels=0,
           check=True):
    """PCG preconditioned by one V-cycle.  Returns (x, iters, hist, status)."""
    lib = _load()
    b = _arr(b, prob.n)
    x = np.zeros(prob.n) if x0 is None else _arr(x0, prob.n).copy()
    hist = np.full(maxit + 1, np.nan)
    iters = ctypes.c_int(-1)
    st = lib.oracle_mg_pcg(*prob._common(), int(nu), float(omega), int(max_levels), _ptr(b),
                           _ptr(x), float(rtol), int(maxit), ctypes.byref(iters), _ptr(hist))
    if check and st not in (OK, ENOTCONV):
        raise OracleError(st, "oracle_mg_pcg")
    return x, iters.value, hist[: max(iters.value, 0) + 1], st
