"""Multigrid preconditioner on the GPU against the CPU oracle.

The tensor-product multigrid (the column solve of eq. (19) as smoother,
horizontal 2x2 coarsening, rediscretised level operators, piecewise-constant
transfers; readings in oracle/oracle_pcg.c) is compared with
oracle.mg_vcycle and oracle.mg_pcg on the same seeded inputs.

Tolerances:
- one V-cycle, 1e-10 relative max-norm.  The GPU and the oracle build
  bitwise-equal level tables and pivots, but the cycle evaluates about
  4*levels stencils and column solves with fused multiply-adds in its own
  order.  The residuals it restricts come from cancelling b - A x with
  ||A x|| up to ~1e5 ||b - A x|| on the strongly anisotropic columns, so
  rounding differences of 1e-16 relative grow to ~1e-12 in the result.  The
  bar leaves two orders of margin above that;
- solves: the iteration count to 1e-10 within one, and the iterate at the
  oracle's count within 1e-8 relative (the solver's parity bar).
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
VC_TOL = 1e-10
SOL_TOL = 1e-8


def case(nx, ny, nz, varying, graded, a_v, seed):
    h = W.layer_thickness(nz, graded)
    ah = W.horizontal_coefficient(nx, ny, varying)
    prob = oracle.Problem(nx, ny, nz, ah=ah, a_v=a_v, mass=1.0, h=h)
    kw = dict(a_h=1.0, a_h_field=ah if varying else None, a_v=a_v, mass=1.0, dz=h)
    b = W.uniform_rhs(prob.n, seed)
    return prob, kw, b


def rel_maxdiff(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


VCYCLE_CASES = [
    # nx, ny, nz, varying, graded, a_v, nu, omega, max_levels
    (16, 16, 12, True, True, 1e3, 1, 0.8, 0),
    (32, 8, 7, False, False, 1e2, 1, 0.8, 0),
    (12, 8, 5, True, False, 1e2, 2, 0.8, 0),      # 12x8 -> 6x4 -> 3x2
    (64, 64, 64, True, True, 1e5, 1, 0.8, 0),     # 7 levels, down to one column
    (40, 36, 33, True, True, 1e4, 1, 1.0, 2),     # two-grid
    (96, 2, 16, False, True, 1e3, 3, 0.7, 0),     # 96x2 -> 48x1
]


@pytest.mark.parametrize("cfg", VCYCLE_CASES, ids=lambda c: "x".join(map(str, c[:3])) +
                         "-nu%d-w%g-L%d" % c[6:9])
def test_vcycle_matches_oracle(cfg):
    nx, ny, nz, varying, graded, a_v, nu, omega, maxl = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v, seed=21)
    z_ref = oracle.mg_vcycle(prob, b, nu=nu, omega=omega, max_levels=maxl)
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_multigrid(nu, omega, maxl)
        s.set_preconditioner("multigrid")
        assert s.multigrid_levels == oracle.mg_levels(nx, ny, maxl)
        z = s.mg_vcycle(torch.from_numpy(b).to(DEV)).cpu().numpy()
    assert rel_maxdiff(z, z_ref) <= VC_TOL


SOLVE_CASES = [
    (32, 32, 16, False, False, 1e2),
    (40, 36, 64, True, True, 1e4),
    (64, 64, 128, True, True, 1e5),
    (24, 10, 130, False, True, 1e3),
]


@pytest.mark.parametrize("cfg", SOLVE_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_mg_solve_matches_oracle(cfg):
    nx, ny, nz, varying, graded, a_v = cfg
    prob, kw, b = case(nx, ny, nz, varying, graded, a_v, seed=22)
    x_ref, it_ref, hist_ref, st_ref = oracle.mg_pcg(prob, b, rtol=1e-10)
    assert st_ref == oracle.OK
    _, it_line, _, _ = oracle.pcg(prob, b, rtol=1e-10)
    assert it_ref < it_line
    with mf.Solver(nx, ny, nz, **kw) as s:
        s.set_preconditioner("multigrid")
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        iters, hist, st = s.solve(bd, x, rtol=1e-10, maxit=500)
        assert st == mf.PCG_OK and abs(iters - it_ref) <= 1
        m = min(iters, it_ref) + 1
        np.testing.assert_allclose(hist[:m], hist_ref[:m], rtol=1e-6, atol=1e-13)
        x.zero_()
        it2, _, st2 = s.solve(bd, x, rtol=0.0, maxit=it_ref)
        assert (it2, st2) == (it_ref, mf.PCG_OK)
        xs = x.cpu().numpy()
    assert np.linalg.norm(xs - x_ref) <= SOL_TOL * np.linalg.norm(x_ref)


def test_mg_solve_is_bitwise_repeatable_and_timed():
    prob, kw, b = case(48, 32, 40, True, True, 1e4, seed=23)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_preconditioner("multigrid")
        s.enable_timing(True)
        bd = torch.from_numpy(b).to(DEV)
        x1, x2 = torch.zeros_like(bd), torch.zeros_like(bd)
        i1, h1, _ = s.solve(bd, x1, rtol=1e-10)
        i2, h2, _ = s.solve(bd, x2, rtol=1e-10)
        t = s.kernel_times()
        info = s.launch_info()
    assert i1 == i2 and np.array_equal(h1, h2) and torch.equal(x1, x2)
    # the V-cycle is timed as the preconditioner step of every iteration
    assert t["precond_fused"][1] >= 2 * (i1 + 1) and t["spmv_fused"][1] >= 2 * i1
    assert info["last_solve_launches"] > 4 * i1


def test_mg_status_semantics():
    prob, kw, b = case(20, 18, 16, True, True, 1e3, seed=24)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_preconditioner("multigrid")
        bd = torch.from_numpy(b).to(DEV)
        _, it_ref, _, _ = oracle.mg_pcg(prob, b, rtol=1e-8)
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-8, maxit=it_ref - 1)
        assert (it, st) == (it_ref - 1, mf.PCG_ENOTCONV)
        x.zero_()
        it, hist, st = s.solve(torch.zeros_like(bd), x, rtol=1e-10)
        assert (it, st) == (0, mf.PCG_OK) and float(x.abs().max()) == 0.0
        bad = bd.clone()
        bad[77] = float("nan")
        x.zero_()
        _, _, st = s.solve(bad, x, rtol=1e-10)
        assert st == mf.PCG_EBREAKDOWN
        # a non-zero initial guess, as in the oracle
        x0 = np.random.default_rng(5).standard_normal(prob.n)
        x.copy_(torch.from_numpy(x0))
        it, _, st = s.solve(bd, x, rtol=1e-9)
        x_ref, it_ref, _, _ = oracle.mg_pcg(prob, b, x0=x0, rtol=1e-9)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        assert np.linalg.norm(x.cpu().numpy() - x_ref) <= 1e-7 * np.linalg.norm(x_ref)


def test_mg_follows_coefficient_updates_and_switches_back():
    prob, kw, b = case(32, 16, 24, True, True, 1e3, seed=25)
    prob2 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=prob.ah * 3.0, a_v=2e4, mass=0.5,
                           h=prob.h)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        s.set_preconditioner("multigrid")
        s.update_coeffs(a_h_field=prob2.ah, a_v=2e4, mass=0.5, dz=prob.h)
        bd = torch.from_numpy(b).to(DEV)
        z = s.mg_vcycle(bd).cpu().numpy()
        assert rel_maxdiff(z, oracle.mg_vcycle(prob2, b)) <= VC_TOL
        x = torch.zeros_like(bd)
        it, _, st = s.solve(bd, x, rtol=1e-10)
        x_ref, it_ref, _, _ = oracle.mg_pcg(prob2, b, rtol=1e-10)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1
        # a constant a_h through the same context
        s.update_coeffs(a_h=0.7, a_v=2e4, mass=0.5, dz=prob.h)
        prob3 = oracle.Problem(prob.nx, prob.ny, prob.nz, ah=0.7, a_v=2e4, mass=0.5, h=prob.h)
        z = s.mg_vcycle(bd).cpu().numpy()
        assert rel_maxdiff(z, oracle.mg_vcycle(prob3, b)) <= VC_TOL
        # back to the column preconditioner: the solve matches line PCG again
        s.set_preconditioner("line")
        assert s.multigrid_levels == 0
        x.zero_()
        it, _, st = s.solve(bd, x, rtol=1e-10)
        _, it_line, _, _ = oracle.pcg(prob3, b, rtol=1e-10)
        assert st == mf.PCG_OK and abs(it - it_line) <= 1


def test_mg_arguments():
    with mf.Solver(7, 8, 6, a_h=1.0, a_v=10.0) as s:      # odd nx: nothing to coarsen
        with pytest.raises(mf.PCGError) as e:
            s.set_preconditioner("multigrid")
        assert e.value.status == mf.PCG_EINVAL
        assert s.multigrid_levels == 0
        with pytest.raises(mf.PCGError):
            s.mg_vcycle(torch.zeros(7 * 8 * 6, dtype=torch.float64, device=DEV))
    with mf.Solver(8, 8, 6, a_h=1.0, a_v=10.0) as s:
        s.set_preconditioner("multigrid")
        assert s.multigrid_levels == 4
        with pytest.raises(mf.PCGError) as e:
            s.set_layout("column")
        assert e.value.status == mf.PCG_EINVAL
        for bad in [(0, 0.8, 0), (1, 0.0, 0), (1, 1.5, 0), (1, 0.8, -1), (1, 0.8, 1)]:
            with pytest.raises(mf.PCGError) as e:
                s.set_multigrid(*bad)
            assert e.value.status == mf.PCG_EINVAL
        s.set_multigrid(2, 0.9, 3)
        assert s.multigrid_levels == 3
        with pytest.raises(mf.PCGError):
            mf.pcg_set_preconditioner(s.ctx, 5)
