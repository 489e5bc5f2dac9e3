"""The preconditioner solve that allocates nothing, checked against pcg_precond
and against the CPU oracle.

pcg_precond_dot_noalloc is for callers that must not allocate device memory
while they run -- code that must not synchronise the device (as cudaFree
does), applications that reserve all device memory for their own pool.  It
returns z = M^{-1} r and
<r, z>, taking its scratch from a fixed array inside the library that every
call reuses.  So it must agree with pcg_precond, and with the oracle's
column solve (eq. (19)) and <r, z> formed from it, on every call, not only
the first, and after the context's coefficients or layout change.  This
file sorts last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import matrix_free_pcg_gb300 as mf  # noqa: E402

DEV = torch.device("cuda:0")
TOL = 1e-12


def rel_maxdiff(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("shape", [(37, 29, 16, True), (64, 48, 64, False), (33, 5, 7, True)])
def test_noalloc_matches_precond_on_two_calls_in_a_row(shape):
    nx, ny, nz, varying = shape
    n = nx * ny * nz
    h = W.layer_thickness(nz, graded=True)
    ah = W.horizontal_coefficient(nx, ny, varying)
    kw = dict(a_h_field=ah if varying else None, a_h=1.0, a_v=1e3, mass=1.0, dz=h)
    rng = np.random.default_rng(nz)
    prob = oracle.Problem(nx, ny, nz, ah=ah if varying else 1.0, a_v=1e3, mass=1.0, h=h)
    with mf.Solver(nx, ny, nz, **kw) as s:
        for call, r_host in enumerate([rng.uniform(-1, 1, n), rng.standard_normal(n)]):
            r = torch.from_numpy(r_host).to(DEV)
            z_lib = s.precond(r).cpu().numpy()
            z_orc = oracle.precond(prob, r_host)
            rz_orc = float(np.dot(r_host, z_orc))
            z = torch.full_like(r, float("nan"))
            rz = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
            mf.pcg_precond_dot_noalloc(s.ctx, n, r, z, rz)
            torch.cuda.synchronize()
            zn = z.cpu().numpy()
            assert rel_maxdiff(zn, z_lib) <= TOL, "call %d: z against pcg_precond" % call
            assert rel_maxdiff(zn, z_orc) <= TOL, "call %d: z against the oracle" % call
            assert abs(float(rz.item()) - rz_orc) <= TOL * abs(rz_orc), "call %d: <r,z>" % call
        # the same input again gives the same bits: nothing left over in the scratch
        z2 = torch.empty_like(r)
        rz2 = torch.empty((1,), dtype=torch.float64, device=DEV)
        mf.pcg_precond_dot_noalloc(s.ctx, n, r, z2, rz2)
        torch.cuda.synchronize()
        assert torch.equal(z2, z) and torch.equal(rz2, rz)


def test_noalloc_rejects_grids_beyond_its_scratch():
    nx, ny, nz = 2048, 1025, 2          # 2,099,200 columns > 65,536 tiles of 32
    with mf.Solver(nx, ny, nz, a_h=1.0, a_v=10.0, mass=1.0) as s:
        n = nx * ny * nz
        r = torch.zeros(n, dtype=torch.float64, device=DEV)
        z = torch.empty_like(r)
        rz = torch.empty((1,), dtype=torch.float64, device=DEV)
        with pytest.raises(mf.PCGError) as e:
            mf.pcg_precond_dot_noalloc(s.ctx, n, r, z, rz)
        assert e.value.status == mf.PCG_EINVAL
        assert "no-allocation scratch" in mf.pcg_last_error(s.ctx)


def test_noalloc_follows_coefficient_and_layout_changes():
    # the entry point reads the context's current tables: a new a_h field and
    # a_v from pcg_update_coeffs, under each solver layout and with the
    # substructured sweep selected, must all be seen
    nx, ny, nz = 40, 24, 32
    n = nx * ny * nz
    h = W.layer_thickness(nz, graded=True)
    ah0 = W.horizontal_coefficient(nx, ny, True)
    ah1 = 0.25 + np.random.default_rng(5).uniform(0.0, 2.0, (ny, nx))
    r_host = np.random.default_rng(6).uniform(-1, 1, n)
    r = torch.from_numpy(r_host).to(DEV)
    with mf.Solver(nx, ny, nz, a_h_field=ah0, a_v=1e3, mass=1.0, dz=h) as s:
        s.update_coeffs(a_h_field=ah1, a_v=2e4, mass=0.5, dz=h)
        prob = oracle.Problem(nx, ny, nz, ah=ah1, a_v=2e4, mass=0.5, h=h)
        z_orc = oracle.precond(prob, r_host)
        rz_orc = float(np.dot(r_host, z_orc))
        for layout, blocks in (("column", 1), ("tiled", 1), ("tiled", 2)):
            s.set_layout(layout)
            s.set_substructuring(blocks)
            z = torch.full_like(r, float("nan"))
            rz = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
            mf.pcg_precond_dot_noalloc(s.ctx, n, r, z, rz)
            z_lib = s.precond(r).cpu().numpy()
            zn = z.cpu().numpy()
            assert rel_maxdiff(zn, z_lib) <= TOL, (layout, blocks)
            assert rel_maxdiff(zn, z_orc) <= TOL, (layout, blocks)
            assert abs(float(rz.item()) - rz_orc) <= TOL * abs(rz_orc), (layout, blocks)


def test_noalloc_rejects_overlapping_arguments():
    nx, ny, nz = 8, 8, 4
    n = nx * ny * nz
    with mf.Solver(nx, ny, nz, a_h=1.0, a_v=10.0, mass=1.0) as s:
        buf = torch.zeros(2 * n + 1, dtype=torch.float64, device=DEV)
        r, z = buf[:n], buf[n:2 * n]
        for rz in (buf[3:4], buf[n + 5:n + 6]):   # inside r, inside z
            with pytest.raises(mf.PCGError) as e:
                mf.pcg_precond_dot_noalloc(s.ctx, n, r, z, rz)
            assert e.value.status == mf.PCG_EINVAL
        with pytest.raises(mf.PCGError):
            mf.pcg_precond_dot_noalloc(s.ctx, n, r, buf[1:n + 1], buf[2 * n:])  # r and z overlap
        mf.pcg_precond_dot_noalloc(s.ctx, n, r, z, buf[2 * n:])  # disjoint: accepted
        # rz just before r, and just before z: one value, not n, so disjoint
        mf.pcg_precond_dot_noalloc(s.ctx, n, buf[1:n + 1], buf[n + 1:], buf[0:1])
        mf.pcg_precond_dot_noalloc(s.ctx, n, buf[n + 1:], buf[1:n + 1], buf[0:1])
        torch.cuda.synchronize()
