"""Pins for the CPU oracle: each check compares it with something the pages
or the mathematics fix independently of its own code (closed forms, a
Kronecker assembly, dense LAPACK solves, scipy's CG, a hand-worked case).

Reference: Mueller et al., "Matrix-free GPU implementation of a
preconditioned conjugate gradient solver for anisotropic elliptic PDEs":
operator section 3 eqs. (3), (5)-(8) and (18); preconditioner section 4.1 and
eq. (19); PCG section 4 and Algorithm 1.
"""
import os

import numpy as np
import pytest
import scipy.linalg as sla
import scipy.sparse.linalg as spla

import oracle
import workloads as W
from tests import tensor_product as tp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def random_problem(nx, ny, nz, seed, graded=True, varying=True, a_v=50.0, mass=1.3):
    rng = np.random.default_rng(seed)
    h = rng.uniform(0.2, 3.0, nz) if graded else np.ones(nz)
    ah = rng.uniform(0.3, 2.0, (ny, nx)) if varying else np.full((ny, nx), 0.7)
    return oracle.Problem(nx, ny, nz, ah=ah, a_v=a_v, mass=mass, h=h), ah, h


def dense_oracle_A(prob):
    n = prob.n
    A = np.empty((n, n))
    for c in range(n):
        e = np.zeros(n)
        e[c] = 1.0
        A[:, c] = oracle.apply_A(prob, e)
    return A


def dense_oracle_Minv(prob):
    n = prob.n
    Minv = np.empty((n, n))
    for c in range(n):
        e = np.zeros(n)
        e[c] = 1.0
        Minv[:, c] = oracle.precond(prob, e)
    return Minv


# ------------------------------------------------------------------ operator

@pytest.mark.parametrize("shape", [(4, 4, 4), (3, 5, 7), (1, 3, 2), (2, 2, 3), (5, 1, 1),
                                   (3, 3, 1)])
def test_operator_equals_tensor_product_assembly(shape):
    nx, ny, nz = shape
    prob, ah, h = random_problem(nx, ny, nz, seed=sum(shape))
    A = dense_oracle_A(prob)
    A_ref = tp.assemble_A(ah, h, prob.a_v, prob.mass).toarray()
    assert np.max(np.abs(A - A_ref)) <= 1e-13 * np.max(np.abs(A_ref))


def test_operator_hand_worked_2x1x2():
    rows = np.loadtxt(os.path.join(GOLDEN, "hand_2x1x2.txt"))
    A_hand, M_hand = rows[:4], rows[4:]
    prob = oracle.Problem(2, 1, 2, ah=np.array([1.0, 2.0]), a_v=2.0, mass=1.0,
                          h=np.array([1.0, 3.0]))
    np.testing.assert_allclose(dense_oracle_A(prob), A_hand, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dense_oracle_Minv(prob), np.linalg.inv(M_hand),
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("pqm", [(0, 0, 0), (1, 0, 0), (0, 2, 1), (3, 1, 4), (2, 3, 2)])
def test_operator_fourier_eigenpairs(pqm):
    nx, ny, nz, a_h, a_v, mass = 8, 6, 5, 0.7, 80.0, 1.3
    p, q, m = pqm
    prob = oracle.Problem(nx, ny, nz, ah=a_h, a_v=a_v, mass=mass)
    v = tp.fourier_mode(nx, ny, nz, p, q, m)
    lam = (mass + a_h * (4 * np.sin(np.pi * p / nx) ** 2 + 4 * np.sin(np.pi * q / ny) ** 2)
           + a_v * 4 * np.sin(np.pi * m / (2 * nz)) ** 2)
    Av = oracle.apply_A(prob, v)
    assert np.max(np.abs(Av - lam * v)) <= 1e-12 * lam * np.max(np.abs(v))


def test_operator_symmetric_and_positive():
    prob, _, _ = random_problem(9, 7, 11, seed=3)
    rng = np.random.default_rng(4)
    x, y = rng.standard_normal(prob.n), rng.standard_normal(prob.n)
    Ax, Ay = oracle.apply_A(prob, x), oracle.apply_A(prob, y)
    assert abs(Ax @ y - x @ Ay) <= 1e-13 * np.linalg.norm(Ax) * np.linalg.norm(y)
    assert x @ Ax > 0 and y @ Ay > 0


def test_operator_row_sums_are_mass_times_thickness():
    prob, ah, h = random_problem(6, 5, 9, seed=5)
    ones = np.ones(prob.n)
    y = oracle.apply_A(prob, ones).reshape(prob.ny, prob.nx, prob.nz)
    A_ref = tp.assemble_A(ah, h, prob.a_v, prob.mass)
    scale = np.asarray(abs(A_ref).sum(axis=1)).reshape(y.shape)
    assert np.all(np.abs(y - prob.mass * h[None, None, :]) <= 1e-14 * scale)


def test_operator_sampled_cells_match_full():
    prob, _, _ = random_problem(7, 6, 5, seed=6)
    x = np.random.default_rng(7).standard_normal(prob.n)
    cells = np.random.default_rng(8).integers(0, prob.n, 50)
    np.testing.assert_array_equal(oracle.apply_A_cells(prob, x, cells),
                                  oracle.apply_A(prob, x)[cells])
    with pytest.raises(oracle.OracleError):
        oracle.apply_A_cells(prob, x, [prob.n])


# ------------------------------------------------------------ preconditioner

@pytest.mark.parametrize("nz", [1, 2, 3, 5, 8, 16])
def test_precond_equals_dense_solve_of_column_blocks(nz):
    prob, ah, h = random_problem(4, 3, nz, seed=10 + nz)
    r = np.random.default_rng(nz).standard_normal(prob.n)
    z = oracle.precond(prob, r)
    A_ref = tp.assemble_A(ah, h, prob.a_v, prob.mass)
    M_def = tp.block_diagonal_part(A_ref, nz).toarray()       # drop column couplings
    M_eq19 = tp.assemble_M(ah, h, prob.a_v, prob.mass).toarray()
    np.testing.assert_allclose(M_def, M_eq19, rtol=1e-14, atol=1e-14)
    z_ref = np.linalg.solve(M_def, r)
    assert np.max(np.abs(z - z_ref)) <= 1e-13 * np.max(np.abs(z_ref))


def test_precond_single_column_matches_banded_lapack():
    nz = 64
    h = W.layer_thickness(nz, graded=True)
    prob = oracle.Problem(1, 1, nz, ah=0.0, a_v=1e5, mass=1.0, h=h)
    r = np.random.default_rng(11).standard_normal(nz)
    t = 1e5 / (0.5 * (h[:-1] + h[1:]))
    main = h.copy()
    main[:-1] += t
    main[1:] += t
    ab = np.zeros((3, nz))
    ab[0, 1:] = -t
    ab[1] = main
    ab[2, :-1] = -t
    z_ref = sla.solve_banded((1, 1), ab, r)
    z = oracle.precond(prob, r)
    assert np.max(np.abs(z - z_ref)) <= 1e-12 * np.max(np.abs(z_ref))


@pytest.mark.parametrize("m", [0, 1, 3])
def test_precond_closed_form_eigenvalue(m):
    nx, ny, nz, a_h, a_v, mass = 5, 4, 6, 0.9, 40.0, 1.1
    prob = oracle.Problem(nx, ny, nz, ah=a_h, a_v=a_v, mass=mass)
    g = np.random.default_rng(m).standard_normal((ny, nx, 1))
    k = np.arange(nz)
    v = (g * np.cos(np.pi * m * (k + 0.5) / nz)[None, None, :]).reshape(-1)
    mu = mass + 4 * a_h + a_v * 4 * np.sin(np.pi * m / (2 * nz)) ** 2
    z = oracle.precond(prob, v)
    assert np.max(np.abs(z - v / mu)) <= 1e-13 * np.max(np.abs(v / mu))


def test_precond_columns_matches_full():
    prob, _, _ = random_problem(6, 4, 7, seed=12)
    r = np.random.default_rng(13).standard_normal(prob.n)
    cols = np.array([0, 5, 23, 11])
    z = oracle.precond(prob, r).reshape(-1, prob.nz)
    np.testing.assert_array_equal(oracle.precond_columns(prob, r, cols), z[cols])


def test_precond_rejects_non_spd_column():
    prob = oracle.Problem(3, 3, 4, ah=1.0, a_v=1.0, mass=-10.0)
    with pytest.raises(oracle.OracleError) as e:
        oracle.precond(prob, np.ones(prob.n))
    assert e.value.status == oracle.EBREAKDOWN


# -------------------------------------------------------------------- solver

def test_pcg_matches_cholesky_solution():
    prob, ah, h = random_problem(4, 4, 4, seed=20)
    A = tp.assemble_A(ah, h, prob.a_v, prob.mass).toarray()
    b = np.random.default_rng(21).standard_normal(prob.n)
    x_ref = sla.cho_solve(sla.cho_factor(A), b)
    x, iters, hist, st = oracle.pcg(prob, b, rtol=1e-14, maxit=200)
    assert st == oracle.OK
    assert np.linalg.norm(x - x_ref) <= 1e-10 * np.linalg.norm(x_ref)
    assert hist[-1] < 1e-14 <= hist[-2]


@pytest.mark.parametrize("k", [1, 2, 5, 9])
def test_pcg_iterates_match_scipy_cg(k):
    """k steps of textbook PCG equal k steps of scipy's CG with the same M."""
    prob, ah, h = random_problem(5, 4, 6, seed=30)
    A = tp.assemble_A(ah, h, prob.a_v, prob.mass)
    M = tp.assemble_M(ah, h, prob.a_v, prob.mass).tocsc()
    Msolve = spla.factorized(M)
    Mop = spla.LinearOperator(A.shape, matvec=Msolve)
    b = np.random.default_rng(31).standard_normal(prob.n)
    x_ref, _ = spla.cg(A, b, x0=np.zeros(prob.n), rtol=1e-300, atol=0.0, maxiter=k, M=Mop)
    x, iters, _, st = oracle.pcg(prob, b, rtol=0.0, maxit=k)
    assert iters == k and st == oracle.OK
    assert np.linalg.norm(x - x_ref) <= 1e-11 * np.linalg.norm(x_ref)


@pytest.mark.parametrize("cfg", [
    # nx, ny, nz, seed, graded, varying, a_v, rtol
    (6, 5, 12, 70, True, True, 1e3, 1e-8),
    (8, 8, 6, 71, False, True, 50.0, 1e-10),
    (5, 7, 9, 72, True, False, 1e4, 1e-6),
    (9, 4, 16, 73, True, True, 1e5, 1e-10),
])
def test_pcg_iteration_count_and_history_match_scipy_cg(cfg):
    """The iteration at which ||r_k|| < rtol ||r_0|| first holds (x0 = 0, so
    ||r_0|| = ||b||), and ||r_k|| / ||r_0|| on the way there, against scipy's
    CG -- its own loop and the same stopping rule -- with the same matrix and
    M; scipy's iterates give the true residuals."""
    nx, ny, nz, seed, graded, varying, a_v, rtol = cfg
    prob, ah, h = random_problem(nx, ny, nz, seed, graded=graded, varying=varying, a_v=a_v)
    A = tp.assemble_A(ah, h, prob.a_v, prob.mass).tocsr()
    M = tp.assemble_M(ah, h, prob.a_v, prob.mass).tocsc()
    Mop = spla.LinearOperator(A.shape, matvec=spla.factorized(M))
    b = np.random.default_rng(seed + 1).standard_normal(prob.n)
    xs = []
    _, info = spla.cg(A, b, x0=np.zeros(prob.n), rtol=rtol, atol=0.0, maxiter=500, M=Mop,
                      callback=lambda xk: xs.append(xk.copy()))
    assert info == 0
    x, iters, hist, st = oracle.pcg(prob, b, rtol=rtol, maxit=500)
    assert st == oracle.OK and iters == len(xs) > 1
    true = np.array([np.linalg.norm(b - A @ xk) for xk in xs]) / np.linalg.norm(b)
    np.testing.assert_allclose(hist[1:], true, rtol=1e-6, atol=1e-12)
    assert hist[iters] < rtol <= hist[iters - 1]


def test_pcg_zero_horizontal_coupling_converges_in_one_iteration():
    prob = oracle.Problem(6, 5, 8, ah=0.0, a_v=1e3, mass=1.0,
                          h=W.layer_thickness(8, graded=True))
    b = np.random.default_rng(40).uniform(-1, 1, prob.n)
    x, iters, hist, st = oracle.pcg(prob, b, rtol=1e-10)
    assert (iters, st) == (1, oracle.OK)
    assert np.linalg.norm(oracle.apply_A(prob, x) - b) <= 1e-12 * np.linalg.norm(b)


def test_pcg_eigenmode_rhs_converges_in_one_iteration():
    nx, ny, nz, a_h, a_v, mass = 8, 6, 5, 1.0, 100.0, 1.0
    prob = oracle.Problem(nx, ny, nz, ah=a_h, a_v=a_v, mass=mass)
    p, q, m = 1, 2, 3
    v = tp.fourier_mode(nx, ny, nz, p, q, m)
    lam = (mass + a_h * (4 * np.sin(np.pi * p / nx) ** 2 + 4 * np.sin(np.pi * q / ny) ** 2)
           + a_v * 4 * np.sin(np.pi * m / (2 * nz)) ** 2)
    x, iters, hist, st = oracle.pcg(prob, v, rtol=1e-10)
    assert (iters, st) == (1, oracle.OK)
    assert np.max(np.abs(x - v / lam)) <= 1e-13 * np.max(np.abs(v / lam))


def test_pcg_stops_after_as_many_iterations_as_distinct_eigenvalues():
    """b in the span of m eigenvectors of M^-1 A with distinct eigenvalues: the
    Krylov space holds the solution after m steps, so PCG stops at exactly m
    (the residual at rounding level there and not before), with x the sum of
    each mode over its eigenvalue of A.  With a constant a_h and uniform
    layers the Fourier x cosine modes are eigenvectors of A and of M alike."""
    nx, ny, nz, a_h, a_v, mass = 8, 6, 5, 1.0, 100.0, 1.0
    prob = oracle.Problem(nx, ny, nz, ah=a_h, a_v=a_v, mass=mass)
    modes = [(1, 2, 3), (2, 0, 1), (4, 3, 0)]

    def eig(p, q, m):  # of A, and of M^-1 A
        lh = 4 * np.sin(np.pi * p / nx) ** 2 + 4 * np.sin(np.pi * q / ny) ** 2
        lv = 4 * np.sin(np.pi * m / (2 * nz)) ** 2
        lam = mass + a_h * lh + a_v * lv
        return lam, lam / (mass + 4 * a_h + a_v * lv)

    assert np.min(np.diff(sorted(eig(*t)[1] for t in modes))) > 1e-2
    for count in (1, 2, 3):
        b = sum(tp.fourier_mode(nx, ny, nz, *t) for t in modes[:count])
        x_ref = sum(tp.fourier_mode(nx, ny, nz, *t) / eig(*t)[0] for t in modes[:count])
        x, iters, hist, st = oracle.pcg(prob, b, rtol=1e-10)
        assert (iters, st) == (count, oracle.OK)
        assert hist[count] < 1e-12 and np.all(hist[:count] > 1e-3)
        assert np.max(np.abs(x - x_ref)) <= 1e-12 * np.max(np.abs(x_ref))


def test_pcg_error_decreases_monotonically_in_A_norm():
    prob, ah, h = random_problem(5, 5, 6, seed=50)
    A = tp.assemble_A(ah, h, prob.a_v, prob.mass).toarray()
    b = np.random.default_rng(51).standard_normal(prob.n)
    x_ref = np.linalg.solve(A, b)
    errs = []
    for k in range(0, 14):
        x, iters, _, _ = oracle.pcg(prob, b, rtol=0.0, maxit=k)
        e = x - x_ref
        errs.append(np.sqrt(e @ A @ e))
    errs = np.array(errs)
    assert np.all(np.diff(errs) < 0), errs
    assert errs[-1] < 1e-4 * errs[0]


def test_pcg_history_and_status_semantics():
    prob, _, _ = random_problem(6, 6, 8, seed=60)
    b = np.random.default_rng(61).standard_normal(prob.n)
    x, iters, hist, st = oracle.pcg(prob, b, rtol=1e-8)
    assert st == oracle.OK and hist[0] == 1.0 and len(hist) == iters + 1
    assert hist[iters] < 1e-8 <= hist[iters - 1]
    r = b - oracle.apply_A(prob, x)
    assert np.linalg.norm(r) / np.linalg.norm(b) < 1e-7
    _, it2, _, st2 = oracle.pcg(prob, b, rtol=1e-8, maxit=iters - 1)
    assert (it2, st2) == (iters - 1, oracle.ENOTCONV)
    _, it3, _, st3 = oracle.pcg(prob, b, rtol=0.0, maxit=3)
    assert (it3, st3) == (3, oracle.OK)
    x0 = np.random.default_rng(62).standard_normal(prob.n)
    _, it4, h4, st4 = oracle.pcg(prob, np.zeros(prob.n), x0=np.zeros(prob.n))
    assert (it4, st4) == (0, oracle.OK) and h4[0] == 0.0
    # restart from a converged iterate: x0 carries the state
    x5, it5, _, st5 = oracle.pcg(prob, b, x0=x0, rtol=1e-8)
    assert st5 == oracle.OK and np.linalg.norm(x5 - x) <= 1e-6 * np.linalg.norm(x)


def test_pcg_manufactured_solution_recovered():
    """b = A u* on the 128x128x64 workload: PCG recovers u*."""
    w = W.WORKLOADS["manufactured_128x128x64"]
    h, ah, ustar = W.make_inputs(w)
    prob = oracle.Problem(w.nx, w.ny, w.nz, ah=ah, a_v=w.a_v, mass=w.mass, h=h)
    b = oracle.apply_A(prob, ustar)
    x, iters, hist, st = oracle.pcg(prob, b, rtol=1e-13, maxit=w.maxit)
    assert st == oracle.OK
    assert np.linalg.norm(x - ustar) <= 1e-9 * np.linalg.norm(ustar)
