"""Python binding of libpcg: matrix-free fp64 PCG for anisotropic 3D
elliptic operators on GB300.

Argument marshalling only.  Every step of the solver runs in the CUDA
kernels of ``libpcg.so`` behind the C ABI of ``include/pcg.h``; PyTorch
provides device memory and streams.  Importing this package loads the
library and raises if it has not been built (``python -m
matrix_free_pcg_gb300.build`` or ``__graft_entry__.build()``): there is no
CPU fallback.

The functions carry the C names (``pcg_create``, ``pcg_apply_A``,
``pcg_precond``, ``pcg_solve``, ...); :class:`Solver` wraps a context.
Vectors are fp64, nx*ny*nz long, vertical index fastest: cell (i, j, k) at
((j*nx)+i)*nz + k, i.e. a contiguous tensor of shape (ny, nx, nz).
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpcg.so")

PCG_OK, PCG_EINVAL, PCG_ENOMEM, PCG_ECUDA, PCG_ENOTCONV, PCG_EBREAKDOWN, PCG_ETIMEOUT = range(7)
STATUS_NAMES = {0: "PCG_OK", 1: "PCG_EINVAL", 2: "PCG_ENOMEM", 3: "PCG_ECUDA",
                4: "PCG_ENOTCONV", 5: "PCG_EBREAKDOWN", 6: "PCG_ETIMEOUT"}
KERNEL_KINDS = ["precond_fused", "spmv_fused", "residual", "finalize", "apply_A", "precond",
                "setup", "loop", "precond_first", "spmv_first"]
PCG_K_COUNT = len(KERNEL_KINDS)

EXPORTED = ["pcg_create", "pcg_destroy", "pcg_update_coeffs", "pcg_set_stream", "pcg_apply_A",
            "pcg_precond", "pcg_solve", "pcg_solve_host", "pcg_last_error",
            "pcg_enable_timing", "pcg_kernel_times", "pcg_launch_info",
            "pcg_precond_dot_noalloc", "pcg_set_layout", "pcg_set_factors",
            "pcg_set_substructuring", "pcg_get_substructuring", "pcg_solve_host_x0",
            "pcg_set_loop", "pcg_get_loop", "pcg_test_barrier_absent", "pcg_set_az_form",
            "pcg_get_az_form", "pcg_set_preconditioner", "pcg_set_multigrid",
            "pcg_get_multigrid", "pcg_mg_vcycle", "pcg_update_solve_host",
            "pcg_measure_fp64_rate", "pcg_test_tensor_memory", "pcg_update_solve_host_async",
            "pcg_host_wait", "pcg_solve_from_zero", "pcg_test_poison_work"]
PCG_LAYOUT_COLUMN, PCG_LAYOUT_TILED = 0, 1
PCG_FACTORS_STORED, PCG_FACTORS_RECOMPUTE = 0, 1
PCG_LOOP_AUTO, PCG_LOOP_BATCHED, PCG_LOOP_PERSISTENT, PCG_LOOP_CLUSTER = 0, 1, 2, 3
PCG_AZ_AUTO, PCG_AZ_STENCIL, PCG_AZ_RESIDUAL = 0, 1, 2
PCG_PREC_LINE, PCG_PREC_MULTIGRID = 0, 1


class pcg_coeffs(ctypes.Structure):
    _fields_ = [("a_h", ctypes.c_double), ("a_h_field", ctypes.POINTER(ctypes.c_double)),
                ("a_v", ctypes.c_double), ("mass", ctypes.c_double),
                ("dz", ctypes.POINTER(ctypes.c_double))]


_dp = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


def _load(path=LIB_PATH):
    if not os.path.exists(path):
        raise ImportError("libpcg.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    sig = {
        "pcg_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(pcg_coeffs), ctypes.POINTER(_vp)]),
        "pcg_destroy": (None, [_vp]),
        "pcg_update_coeffs": (ctypes.c_int, [_vp, ctypes.POINTER(pcg_coeffs)]),
        "pcg_set_stream": (ctypes.c_int, [_vp, _vp]),
        "pcg_apply_A": (ctypes.c_int, [_vp, _vp, _vp]),
        "pcg_precond": (ctypes.c_int, [_vp, _vp, _vp]),
        "pcg_solve": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_double, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_solve_from_zero": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_double, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_solve_host": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_double, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_solve_host_x0": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_double, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_update_solve_host": (ctypes.c_int, [_vp, ctypes.POINTER(pcg_coeffs), _vp, _vp, _vp,
                                                 ctypes.c_double, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_update_solve_host_async": (ctypes.c_int, [_vp, ctypes.POINTER(pcg_coeffs), _vp, _vp,
                                                       _vp, ctypes.c_double, ctypes.c_int,
                                                       ctypes.POINTER(ctypes.c_int), _vp]),
        "pcg_host_wait": (ctypes.c_int, [_vp]),
        "pcg_last_error": (ctypes.c_char_p, [_vp]),
        "pcg_enable_timing": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_kernel_times": (ctypes.c_int, [_vp, _vp, _vp]),
        "pcg_launch_info": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_longlong)]),
        "pcg_precond_dot_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
        "pcg_set_layout": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_set_factors": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_set_substructuring": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_get_substructuring": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int)]),
        "pcg_set_loop": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_get_loop": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int)]),
        "pcg_set_az_form": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_set_preconditioner": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_set_multigrid": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_double, ctypes.c_int]),
        "pcg_get_multigrid": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int)]),
        "pcg_mg_vcycle": (ctypes.c_int, [_vp, ctypes.c_void_p, ctypes.c_void_p]),
        "pcg_get_az_form": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int)]),
        "pcg_test_barrier_absent": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_test_tensor_memory": (ctypes.c_int, [_vp, ctypes.c_int]),
        "pcg_test_poison_work": (ctypes.c_int, [_vp]),
        "pcg_measure_fp64_rate": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


class PCGError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), msg))
        self.status = status


def _check(status, ctx=None):
    if status != PCG_OK:
        raise PCGError(status, pcg_last_error(ctx))
    return status


def _f64(a, n, what):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.size != n:
        raise ValueError("%s: expected %d values, got %d" % (what, n, a.size))
    return a


def _dev_ptr(t, n, what):
    """Device pointer of a contiguous fp64 CUDA tensor with n elements."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor on a CUDA device" % what)
    if t.dtype != torch.float64 or not t.is_cuda or not t.is_contiguous() or t.numel() != n:
        raise ValueError("%s must be a contiguous float64 CUDA tensor with %d elements "
                         "(got %s %s %s)" % (what, n, t.dtype, t.device, tuple(t.shape)))
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(a, n, what, writable=False):
    """Host pointer of a C-contiguous fp64 numpy array or CPU tensor with n elements."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda or a.dtype != torch.float64 or not a.is_contiguous() or a.numel() != n:
                raise ValueError("%s must be a contiguous float64 CPU tensor with %d elements"
                                 % (what, n))
            return ctypes.c_void_p(a.data_ptr())
    except ImportError:
        pass
    if not (isinstance(a, np.ndarray) and a.dtype == np.float64 and a.flags.c_contiguous
            and a.size == n and (a.flags.writeable or not writable)):
        raise ValueError("%s must be a C-contiguous float64 array with %d elements" % (what, n))
    return ctypes.c_void_p(a.ctypes.data)


def make_coeffs(nx, ny, nz, a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None):
    """pcg_coeffs plus the numpy arrays it points into (keep both alive)."""
    keep = []
    c = pcg_coeffs()
    c.a_h = float(a_h)
    c.a_v = float(a_v)
    c.mass = float(mass)
    if a_h_field is not None:
        f = _f64(a_h_field, nx * ny, "a_h_field")
        keep.append(f)
        c.a_h_field = f.ctypes.data_as(_dp)
    if dz is not None:
        d = _f64(dz, nz, "dz")
        keep.append(d)
        c.dz = d.ctypes.data_as(_dp)
    return c, keep


# ------------------------------------------------------------ C-named calls

def pcg_last_error(ctx=None):
    return _lib.pcg_last_error(ctx).decode()


def pcg_create(nx, ny, nz, a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None):
    c, keep = make_coeffs(nx, ny, nz, a_h, a_h_field, a_v, mass, dz)
    ctx = ctypes.c_void_p()
    _check(_lib.pcg_create(int(nx), int(ny), int(nz), ctypes.byref(c), ctypes.byref(ctx)))
    return ctx


def pcg_destroy(ctx):
    _lib.pcg_destroy(ctx)


def pcg_update_coeffs(ctx, nx, ny, nz, a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None):
    c, keep = make_coeffs(nx, ny, nz, a_h, a_h_field, a_v, mass, dz)
    return _check(_lib.pcg_update_coeffs(ctx, ctypes.byref(c)), ctx)


def pcg_set_stream(ctx, stream):
    """stream: a torch.cuda.Stream, a raw cudaStream_t integer, or None."""
    handle = getattr(stream, "cuda_stream", stream)
    return _check(_lib.pcg_set_stream(ctx, ctypes.c_void_p(handle or 0)), ctx)


def pcg_set_layout(ctx, layout):
    """PCG_LAYOUT_TILED (default) or PCG_LAYOUT_COLUMN for the solver's internal vectors."""
    return _check(_lib.pcg_set_layout(ctx, int(layout)), ctx)


def pcg_set_factors(ctx, mode):
    """PCG_FACTORS_STORED (default) or PCG_FACTORS_RECOMPUTE: per-cell factors of an
    a_h field read from arrays, or rebuilt in every sweep (row-tiled layout)."""
    return _check(_lib.pcg_set_factors(ctx, int(mode)), ctx)


def pcg_set_substructuring(ctx, nblocks):
    """Blocks per column of the substructured preconditioner solve (row-tiled
    layout): 0 automatic (default), 1 off (Thomas), 2, 4, 8 or 16."""
    return _check(_lib.pcg_set_substructuring(ctx, int(nblocks)), ctx)


def pcg_get_substructuring(ctx):
    """Blocks per column in use by the row-tiled preconditioner sweep (1: Thomas)."""
    v = ctypes.c_int(0)
    _check(_lib.pcg_get_substructuring(ctx, ctypes.byref(v)), ctx)
    return v.value


def pcg_set_loop(ctx, mode):
    """PCG_LOOP_AUTO (default), PCG_LOOP_BATCHED, PCG_LOOP_PERSISTENT or PCG_LOOP_CLUSTER."""
    return _check(_lib.pcg_set_loop(ctx, int(mode)), ctx)


def pcg_get_loop(ctx):
    """The loop the next solve runs: PCG_LOOP_BATCHED, PCG_LOOP_PERSISTENT or PCG_LOOP_CLUSTER."""
    v = ctypes.c_int(0)
    _check(_lib.pcg_get_loop(ctx, ctypes.byref(v)), ctx)
    return v.value


def pcg_set_az_form(ctx, form):
    """PCG_AZ_AUTO (default), PCG_AZ_STENCIL or PCG_AZ_RESIDUAL."""
    return _check(_lib.pcg_set_az_form(ctx, int(form)), ctx)


def pcg_get_az_form(ctx):
    """The form of A z the next solve uses: PCG_AZ_STENCIL or PCG_AZ_RESIDUAL."""
    v = ctypes.c_int(0)
    _check(_lib.pcg_get_az_form(ctx, ctypes.byref(v)), ctx)
    return v.value


def pcg_set_preconditioner(ctx, prec):
    """PCG_PREC_LINE (default) or PCG_PREC_MULTIGRID."""
    return _check(_lib.pcg_set_preconditioner(ctx, int(prec)), ctx)


def pcg_set_multigrid(ctx, nu=1, omega=0.8, max_levels=0):
    """Smoothing steps per side, damping, level cap (0: none)."""
    return _check(_lib.pcg_set_multigrid(ctx, int(nu), float(omega), int(max_levels)), ctx)


def pcg_get_multigrid(ctx):
    """Levels of the multigrid preconditioner in use (0: not selected)."""
    v = ctypes.c_int(0)
    _check(_lib.pcg_get_multigrid(ctx, ctypes.byref(v)), ctx)
    return v.value


def pcg_mg_vcycle(ctx, n, r, z):
    """z = B r, one V-cycle (device tensors of n values, caller's layout)."""
    return _check(_lib.pcg_mg_vcycle(ctx, _dev_ptr(r, n, "r"), _dev_ptr(z, n, "z")), ctx)


def pcg_test_barrier_absent(ctx, absent):
    """Test hook: the persistent loop's barriers miss `absent` arrivals, so the
    next persistent solve's first barrier wait runs out (PCG_ETIMEOUT)."""
    return _check(_lib.pcg_test_barrier_absent(ctx, int(absent)), ctx)


def pcg_test_poison_work(ctx):
    """Test hook: fills the context's work vectors with NaN (as memory left by
    an earlier user may hold); a solve must not depend on what they held."""
    return _check(_lib.pcg_test_poison_work(ctx), ctx)


def pcg_test_tensor_memory(ctx, enable):
    """Test hook: enable=False makes pcg_precond and the column layout's sweep
    keep w in global memory instead of the SM's tensor memory (True: default)."""
    return _check(_lib.pcg_test_tensor_memory(ctx, int(bool(enable))), ctx)


def pcg_apply_A(ctx, n, x, y):
    return _check(_lib.pcg_apply_A(ctx, _dev_ptr(x, n, "x"), _dev_ptr(y, n, "y")), ctx)


def pcg_precond(ctx, n, r, z):
    return _check(_lib.pcg_precond(ctx, _dev_ptr(r, n, "r"), _dev_ptr(z, n, "z")), ctx)


def pcg_solve(ctx, n, b, x, rtol, maxit, history=True, from_zero=False):
    """Returns (iters, hist or None, status); raises on EINVAL/ENOMEM/ECUDA.
    from_zero: pcg_solve_from_zero (x0 = 0; x is written, never read)."""
    it = ctypes.c_int(-1)
    hist = np.full(int(maxit) + 1, np.nan) if history else None
    fn = _lib.pcg_solve_from_zero if from_zero else _lib.pcg_solve
    st = fn(ctx, _dev_ptr(b, n, "b"), _dev_ptr(x, n, "x"), float(rtol), int(maxit),
            ctypes.byref(it), hist.ctypes.data_as(_vp) if history else None)
    if st not in (PCG_OK, PCG_ENOTCONV, PCG_EBREAKDOWN):
        _check(st, ctx)
    return it.value, (hist[: it.value + 1] if history else None), st


def pcg_solve_host(ctx, n, b, x, rtol, maxit, history=True):
    """b, x: host arrays (numpy or CPU tensors, pinned for full speed)."""
    it = ctypes.c_int(-1)
    hist = np.full(int(maxit) + 1, np.nan) if history else None
    st = _lib.pcg_solve_host(ctx, _host_ptr(b, n, "b"), _host_ptr(x, n, "x", writable=True),
                             float(rtol), int(maxit), ctypes.byref(it),
                             hist.ctypes.data_as(_vp) if history else None)
    if st not in (PCG_OK, PCG_ENOTCONV, PCG_EBREAKDOWN):
        _check(st, ctx)
    return it.value, (hist[: it.value + 1] if history else None), st


def pcg_solve_host_x0(ctx, n, b, x0, x, rtol, maxit, history=True):
    """b, x0, x: host arrays; x0 None means a zero initial guess (x is then
    written only)."""
    it = ctypes.c_int(-1)
    hist = np.full(int(maxit) + 1, np.nan) if history else None
    x0p = None if x0 is None else _host_ptr(x0, n, "x0")
    st = _lib.pcg_solve_host_x0(ctx, _host_ptr(b, n, "b"), x0p, _host_ptr(x, n, "x", writable=True),
                                float(rtol), int(maxit), ctypes.byref(it),
                                hist.ctypes.data_as(_vp) if history else None)
    if st not in (PCG_OK, PCG_ENOTCONV, PCG_EBREAKDOWN):
        _check(st, ctx)
    return it.value, (hist[: it.value + 1] if history else None), st


def pcg_update_solve_host(ctx, nx, ny, nz, b, x0, x, rtol, maxit, history=True, a_h=1.0,
                          a_h_field=None, a_v=1.0, mass=1.0, dz=None):
    """New coefficients, then a solve from host arrays b, x0 (None: zero
    initial guess) into x, in one call (b and x0 are copied in while the
    set-up runs)."""
    n = int(nx) * int(ny) * int(nz)
    c, keep = make_coeffs(nx, ny, nz, a_h, a_h_field, a_v, mass, dz)
    it = ctypes.c_int(-1)
    hist = np.full(int(maxit) + 1, np.nan) if history else None
    x0p = None if x0 is None else _host_ptr(x0, n, "x0")
    st = _lib.pcg_update_solve_host(ctx, ctypes.byref(c), _host_ptr(b, n, "b"), x0p,
                                    _host_ptr(x, n, "x", writable=True), float(rtol), int(maxit),
                                    ctypes.byref(it), hist.ctypes.data_as(_vp) if history else None)
    del keep
    if st not in (PCG_OK, PCG_ENOTCONV, PCG_EBREAKDOWN):
        _check(st, ctx)
    return it.value, (hist[: it.value + 1] if history else None), st


def pcg_update_solve_host_async(ctx, nx, ny, nz, b, x0, x, rtol, maxit, history=True, a_h=1.0,
                                a_h_field=None, a_v=1.0, mass=1.0, dz=None):
    """As pcg_update_solve_host, with x's copy to the host left running (it
    overlaps the next call); read x only after pcg_host_wait."""
    n = int(nx) * int(ny) * int(nz)
    c, keep = make_coeffs(nx, ny, nz, a_h, a_h_field, a_v, mass, dz)
    it = ctypes.c_int(-1)
    hist = np.full(int(maxit) + 1, np.nan) if history else None
    x0p = None if x0 is None else _host_ptr(x0, n, "x0")
    st = _lib.pcg_update_solve_host_async(ctx, ctypes.byref(c), _host_ptr(b, n, "b"), x0p,
                                          _host_ptr(x, n, "x", writable=True), float(rtol),
                                          int(maxit), ctypes.byref(it),
                                          hist.ctypes.data_as(_vp) if history else None)
    del keep
    if st not in (PCG_OK, PCG_ENOTCONV, PCG_EBREAKDOWN):
        _check(st, ctx)
    return it.value, (hist[: it.value + 1] if history else None), st


def pcg_host_wait(ctx):
    """Wait for the solution copies left running by pcg_update_solve_host_async."""
    return _check(_lib.pcg_host_wait(ctx), ctx)


def pcg_precond_dot_noalloc(ctx, n, r, z, rz):
    """z = M^{-1} r and rz[0] = <r, z>, with no device allocation.

    For callers that must not allocate device memory while they run (no
    synchronising cudaFree, stream capture in progress, a pre-reserved memory
    pool).  r, z: contiguous float64 CUDA tensors of n values; rz: a float64
    CUDA tensor of one value.  Scratch comes from a fixed array inside the
    library, shared by every call: calls that overlap on the GPU race.  Grids
    above 2,097,152 columns are rejected.
    """
    return _check(_lib.pcg_precond_dot_noalloc(ctx, _dev_ptr(r, n, "r"), _dev_ptr(z, n, "z"),
                                               _dev_ptr(rz, 1, "rz")), ctx)


def pcg_enable_timing(ctx, enable=True):
    return _check(_lib.pcg_enable_timing(ctx, int(bool(enable))), ctx)


def pcg_kernel_times(ctx):
    ms = (ctypes.c_double * PCG_K_COUNT)()
    cnt = (ctypes.c_longlong * PCG_K_COUNT)()
    _check(_lib.pcg_kernel_times(ctx, ms, cnt), ctx)
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def pcg_launch_info(ctx):
    gm, ga, nl = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
    _check(_lib.pcg_launch_info(ctx, ctypes.byref(gm), ctypes.byref(ga), ctypes.byref(nl)), ctx)
    return {"grid_precond": gm.value, "grid_spmv": ga.value, "last_solve_launches": nl.value}


def pcg_measure_fp64_rate(warps_per_sm=32, launches=3):
    """Measured fp64 rate of the current device's non-tensor pipe: a dict with
    lane operations per second (an FMA counts one), the SM clock measured
    inside the fastest launch, and lane operations per SM per clock."""
    rate, mhz, per_clk = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(_lib.pcg_measure_fp64_rate(int(warps_per_sm), int(launches), ctypes.byref(rate),
                                      ctypes.byref(mhz), ctypes.byref(per_clk)))
    return {"lane_ops_per_s": rate.value, "sm_mhz": mhz.value,
            "lanes_per_sm_clk": per_clk.value, "warps_per_sm": int(warps_per_sm),
            "launches": int(launches)}


# ------------------------------------------------------------------- class

class Solver:
    """One solver context on the current CUDA device.

    a_h: constant horizontal coefficient, or a_h_field: (ny, nx) array of
    a_h(i, j); a_v: vertical coefficient; mass: zero-order coefficient;
    dz: nz layer thicknesses (bottom first), default all ones.
    """

    def __init__(self, nx, ny, nz, a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None,
                 stream=None):
        self.nx, self.ny, self.nz = int(nx), int(ny), int(nz)
        self.n = self.nx * self.ny * self.nz
        self.ctx = pcg_create(nx, ny, nz, a_h, a_h_field, a_v, mass, dz)
        if stream is not None:
            pcg_set_stream(self.ctx, stream)

    def close(self):
        if self.ctx is not None:
            pcg_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def update_coeffs(self, a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None):
        pcg_update_coeffs(self.ctx, self.nx, self.ny, self.nz, a_h, a_h_field, a_v, mass, dz)

    def set_stream(self, stream):
        pcg_set_stream(self.ctx, stream)

    def set_layout(self, layout):
        """"column" / PCG_LAYOUT_COLUMN or "tiled" / PCG_LAYOUT_TILED."""
        if isinstance(layout, str):
            layout = {"column": PCG_LAYOUT_COLUMN, "tiled": PCG_LAYOUT_TILED}[layout]
        pcg_set_layout(self.ctx, layout)

    def set_substructuring(self, nblocks):
        """0 automatic, 1 off, or 2/4/8/16 blocks per column."""
        pcg_set_substructuring(self.ctx, nblocks)

    def set_loop(self, mode):
        """"auto", "batched", "persistent" or "cluster" (or the PCG_LOOP_* values)."""
        if isinstance(mode, str):
            mode = {"auto": PCG_LOOP_AUTO, "batched": PCG_LOOP_BATCHED,
                    "persistent": PCG_LOOP_PERSISTENT, "cluster": PCG_LOOP_CLUSTER}[mode]
        pcg_set_loop(self.ctx, mode)

    def set_preconditioner(self, prec):
        """"line" (column solve, default) or "multigrid" (or the PCG_PREC_* values)."""
        if isinstance(prec, str):
            prec = {"line": PCG_PREC_LINE, "multigrid": PCG_PREC_MULTIGRID}[prec]
        pcg_set_preconditioner(self.ctx, prec)

    def set_multigrid(self, nu=1, omega=0.8, max_levels=0):
        pcg_set_multigrid(self.ctx, nu, omega, max_levels)

    @property
    def multigrid_levels(self):
        """Levels of the multigrid preconditioner in use (0: not selected)."""
        return pcg_get_multigrid(self.ctx)

    def mg_vcycle(self, r, z=None):
        """z = B r, one V-cycle on device fp64 tensors of N values."""
        import torch
        if z is None:
            z = torch.empty_like(r)
        pcg_mg_vcycle(self.ctx, self.n, r, z)
        return z

    def set_az_form(self, form):
        """"auto", "stencil" or "residual" (or the PCG_AZ_* values)."""
        if isinstance(form, str):
            form = {"auto": PCG_AZ_AUTO, "stencil": PCG_AZ_STENCIL,
                    "residual": PCG_AZ_RESIDUAL}[form]
        pcg_set_az_form(self.ctx, form)

    @property
    def az_form(self):
        """"stencil" or "residual": how the next solve's stencil sweeps form A z."""
        return {PCG_AZ_STENCIL: "stencil", PCG_AZ_RESIDUAL: "residual"}[
            pcg_get_az_form(self.ctx)]

    @property
    def loop(self):
        """"batched", "persistent" or "cluster": the loop the next solve runs."""
        return {PCG_LOOP_BATCHED: "batched", PCG_LOOP_PERSISTENT: "persistent",
                PCG_LOOP_CLUSTER: "cluster"}[pcg_get_loop(self.ctx)]

    @property
    def substructuring(self):
        """Blocks per column in use (after the automatic choice)."""
        return pcg_get_substructuring(self.ctx)

    def set_factors(self, mode):
        """"stored" / PCG_FACTORS_STORED or "recompute" / PCG_FACTORS_RECOMPUTE."""
        if isinstance(mode, str):
            mode = {"stored": PCG_FACTORS_STORED, "recompute": PCG_FACTORS_RECOMPUTE}[mode]
        pcg_set_factors(self.ctx, mode)

    def apply_A(self, x, y=None):
        import torch
        if y is None:
            y = torch.empty_like(x)
        pcg_apply_A(self.ctx, self.n, x, y)
        return y

    def precond(self, r, z=None):
        import torch
        if z is None:
            z = torch.empty_like(r)
        pcg_precond(self.ctx, self.n, r, z)
        return z

    def solve(self, b, x, rtol=1e-10, maxit=500, history=True):
        """x (device tensor): initial guess in, solution out.
        Returns (iters, residual history, status)."""
        return pcg_solve(self.ctx, self.n, b, x, rtol, maxit, history)

    def solve_from_zero(self, b, x, rtol=1e-10, maxit=500, history=True):
        """pcg_solve_from_zero: x0 = 0; x (device tensor) receives the
        solution and is never read."""
        return pcg_solve(self.ctx, self.n, b, x, rtol, maxit, history, from_zero=True)

    def solve_host(self, b, x, rtol=1e-10, maxit=500, history=True, x0="x"):
        """x0="x": x holds the initial guess (pcg_solve_host); None: zero initial
        guess; or a separate host array (pcg_solve_host_x0)."""
        if isinstance(x0, str) and x0 == "x":
            return pcg_solve_host(self.ctx, self.n, b, x, rtol, maxit, history)
        return pcg_solve_host_x0(self.ctx, self.n, b, x0, x, rtol, maxit, history)

    def update_solve_host(self, b, x, rtol=1e-10, maxit=500, history=True, x0=None, a_h=1.0,
                          a_h_field=None, a_v=1.0, mass=1.0, dz=None):
        """pcg_update_solve_host: new coefficients, then a solve from host
        arrays (b and x0 copied in while the set-up runs)."""
        return pcg_update_solve_host(self.ctx, self.nx, self.ny, self.nz, b, x0, x, rtol, maxit,
                                     history, a_h, a_h_field, a_v, mass, dz)

    def update_solve_host_async(self, b, x, rtol=1e-10, maxit=500, history=True, x0=None,
                                a_h=1.0, a_h_field=None, a_v=1.0, mass=1.0, dz=None):
        """pcg_update_solve_host_async: as update_solve_host, x's copy left
        running; call host_wait before reading x."""
        return pcg_update_solve_host_async(self.ctx, self.nx, self.ny, self.nz, b, x0, x, rtol,
                                           maxit, history, a_h, a_h_field, a_v, mass, dz)

    def host_wait(self):
        pcg_host_wait(self.ctx)

    def enable_timing(self, enable=True):
        pcg_enable_timing(self.ctx, enable)

    def kernel_times(self):
        return pcg_kernel_times(self.ctx)

    def launch_info(self):
        return pcg_launch_info(self.ctx)
