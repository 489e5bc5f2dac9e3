"""Pins of the oracle's tensor-product multigrid (CPU only).

The paper (Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
sections 1, 2 and 9) names the column solve of eq. (19) as the smoother of a
geometric multigrid that coarsens only horizontally (the tensor-product idea
of Boerm and Hiptmair) and leaves the intergrid operators open.  The readings
(2x2 column merging, rediscretised level operators on cells of area 4^l,
piecewise-constant P, R = P^T, damped line relaxation, symmetric V-cycle)
are pinned here against constructions that share nothing with the oracle's
code: Kronecker assemblies from face lists, index-map prolongation matrices,
dense linear algebra for the cycle, and properties every correct V-cycle
preconditioner has.
"""
import numpy as np
import pytest
import scipy.sparse.linalg as spla

import oracle
import workloads as W
from tensor_product import assemble_A, assemble_M, piecewise_constant_prolongation

RNG = np.random.default_rng(2024)


def problem(nx, ny, nz, varying=True, graded=True, a_v=1e3, mass=1.0, ah_scale=1.0):
    h = W.layer_thickness(nz, graded)
    if varying:
        ah = ah_scale * (1.0 + 0.5 * RNG.uniform(-1, 1, (ny, nx)))
    else:
        ah = np.full((ny, nx), ah_scale)
    return oracle.Problem(nx, ny, nz, ah=ah, a_v=a_v, mass=mass, h=h)


def test_level_count():
    assert oracle.mg_levels(32, 32) == 6          # 32 -> 16 -> 8 -> 4 -> 2 -> 1
    assert oracle.mg_levels(12, 8) == 3           # 12x8 -> 6x4 -> 3x2
    assert oracle.mg_levels(7, 8) == 1
    assert oracle.mg_levels(2, 2) == 2
    assert oracle.mg_levels(1024, 1024) == 11
    assert oracle.mg_levels(1024, 1024, max_levels=4) == 4
    assert oracle.mg_levels(64, 16) == 5          # 64x16 -> ... -> 4x1


def test_coarse_ah_is_the_mean_of_the_merged_columns():
    prob = problem(8, 4, 3)
    ah = prob.ah.reshape(4, 8)
    c1 = ah.reshape(2, 2, 4, 2).mean(axis=(1, 3))
    c2 = c1.reshape(1, 2, 2, 2).mean(axis=(1, 3))
    np.testing.assert_allclose(oracle.mg_level_ah(prob, 1), c1, rtol=1e-15)
    np.testing.assert_allclose(oracle.mg_level_ah(prob, 2), c2, rtol=1e-15)
    np.testing.assert_array_equal(oracle.mg_level_ah(prob, 0), ah)


@pytest.mark.parametrize("shape", [(8, 8, 5), (6, 4, 3), (4, 2, 6), (2, 2, 4)])
@pytest.mark.parametrize("level", [1, 2])
def test_level_operator_is_the_rediscretised_assembly(shape, level):
    nx, ny, nz = shape
    if oracle.mg_levels(nx, ny) <= level:
        pytest.skip("no such level")
    prob = problem(nx, ny, nz, a_v=1e2)
    ahc = oracle.mg_level_ah(prob, level)
    nyc, nxc = ahc.shape
    area = 4.0 ** level
    coarse = oracle.Problem(nxc, nyc, nz, ah=ahc, a_v=prob.a_v, mass=prob.mass, h=prob.h)
    A = assemble_A(ahc, prob.h, prob.a_v, prob.mass, area=area)
    for _ in range(3):
        x = RNG.standard_normal(coarse.n)
        y = oracle.apply_A_area(coarse, x, area)
        ref = A @ x
        assert np.max(np.abs(y - ref)) <= 1e-13 * np.max(np.abs(ref))


def test_prolongation_is_piecewise_constant_and_restriction_its_transpose():
    nx, ny, nz = 6, 4, 3
    P = piecewise_constant_prolongation(nx, ny, nz)
    e = RNG.standard_normal(P.shape[1])
    x0 = RNG.standard_normal(P.shape[0])
    np.testing.assert_array_equal(oracle.mg_prolong_add(nx, ny, nz, e, x0), x0 + P @ e)
    r = RNG.standard_normal(P.shape[0])
    np.testing.assert_allclose(oracle.mg_restrict(nx, ny, nz, r), P.T @ r, rtol=1e-15, atol=0)


def test_galerkin_product_doubles_the_horizontal_part_for_constant_ah():
    # with piecewise-constant transfers, R A_f P keeps the vertical and
    # zero-order terms of the rediscretised operator (area 4) and counts the
    # horizontal couplings twice (two fine faces per coarse face)
    nx, ny, nz = 8, 6, 5
    prob = problem(nx, ny, nz, varying=False, a_v=50.0, ah_scale=1.3)
    coarse = oracle.Problem(nx // 2, ny // 2, nz, ah=1.3, a_v=prob.a_v, mass=prob.mass, h=prob.h)
    no_h = oracle.Problem(nx // 2, ny // 2, nz, ah=0.0, a_v=prob.a_v, mass=prob.mass, h=prob.h)
    x = RNG.standard_normal(coarse.n)
    Px = oracle.mg_prolong_add(nx, ny, nz, x, np.zeros(prob.n))
    galerkin = oracle.mg_restrict(nx, ny, nz, oracle.apply_A(prob, Px))
    redisc = oracle.apply_A_area(coarse, x, 4.0)
    vert = oracle.apply_A_area(no_h, x, 4.0)
    np.testing.assert_allclose(galerkin, 2.0 * redisc - vert, rtol=1e-12,
                               atol=1e-12 * np.max(np.abs(galerkin)))


def dense_vcycle(prob, nu, omega, max_levels=0):
    """B as a dense matrix: the V-cycle recursion written with the assembled
    level matrices and library solves."""
    L = oracle.mg_levels(prob.nx, prob.ny, max_levels)
    lev = []
    ah = prob.ah.reshape(prob.ny, prob.nx)
    nx, ny = prob.nx, prob.ny
    for l in range(L):
        if l > 0:
            ah = ah.reshape(ny // 2, 2, nx // 2, 2).mean(axis=(1, 3))
            nx, ny = nx // 2, ny // 2
        area = 4.0 ** l
        A = assemble_A(ah, prob.h, prob.a_v, prob.mass, area=area).toarray()
        M = assemble_M(ah, prob.h, prob.a_v, prob.mass, area=area).toarray()
        P = (piecewise_constant_prolongation(nx, ny, prob.nz).toarray() if l < L - 1 else None)
        lev.append((A, M, P))

    def V(l, b):
        A, M, P = lev[l]
        x = np.zeros_like(b)
        for _ in range(nu):
            x = x + omega * np.linalg.solve(M, b - A @ x)
        if l == L - 1:
            return x
        x = x + P @ V(l + 1, P.T @ (b - A @ x))
        for _ in range(nu):
            x = x + omega * np.linalg.solve(M, b - A @ x)
        return x

    n = prob.n
    return np.column_stack([V(0, np.eye(n)[:, c]) for c in range(n)])


@pytest.mark.parametrize("shape,nu,omega", [((4, 4, 3), 1, 0.8), ((4, 2, 5), 2, 0.8),
                                            ((8, 4, 2), 1, 1.0), ((6, 2, 3), 1, 0.7)])
def test_vcycle_matches_the_dense_recursion(shape, nu, omega):
    nx, ny, nz = shape
    prob = problem(nx, ny, nz, a_v=30.0)
    B = dense_vcycle(prob, nu, omega)
    for _ in range(3):
        r = RNG.standard_normal(prob.n)
        z = oracle.mg_vcycle(prob, r, nu=nu, omega=omega)
        ref = B @ r
        assert np.max(np.abs(z - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_level_cap_two_grid():
    prob = problem(8, 8, 3, a_v=20.0)
    B = dense_vcycle(prob, 1, 0.8, max_levels=2)
    r = RNG.standard_normal(prob.n)
    z = oracle.mg_vcycle(prob, r, max_levels=2)
    np.testing.assert_allclose(z, B @ r, rtol=1e-11, atol=1e-12 * np.max(np.abs(z)))


@pytest.mark.parametrize("nu,omega", [(1, 0.8), (2, 0.8), (1, 1.0)])
def test_vcycle_is_symmetric_positive_definite(nu, omega):
    prob = problem(16, 8, 12, a_v=1e4)
    for _ in range(3):
        x, y = RNG.standard_normal(prob.n), RNG.standard_normal(prob.n)
        bx = oracle.mg_vcycle(prob, x, nu=nu, omega=omega)
        by = oracle.mg_vcycle(prob, y, nu=nu, omega=omega)
        lhs, rhs = bx @ y, x @ by
        assert abs(lhs - rhs) <= 1e-12 * np.linalg.norm(bx) * np.linalg.norm(y)
        assert x @ bx > 0.0


def test_without_horizontal_coupling_the_cycle_is_the_exact_inverse():
    # a_h = 0: M = A on every level, so undamped line relaxation solves at
    # once and the coarse correction is zero
    prob = problem(8, 4, 9, varying=False, ah_scale=0.0, a_v=1e3)
    A = assemble_A(np.zeros((4, 8)), prob.h, prob.a_v, prob.mass)
    b = RNG.standard_normal(prob.n)
    z = oracle.mg_vcycle(prob, b, nu=1, omega=1.0)
    ref = spla.spsolve(A.tocsc(), b)
    assert np.max(np.abs(z - ref)) <= 1e-12 * np.max(np.abs(ref))
    x, it, hist, st = oracle.mg_pcg(prob, b, rtol=1e-12, omega=1.0)
    assert (it, st) == (1, oracle.OK)


def test_mg_pcg_solves_the_system():
    prob = problem(8, 8, 6, a_v=1e3)
    A = assemble_A(prob.ah.reshape(8, 8), prob.h, prob.a_v, prob.mass)
    b = RNG.uniform(-1, 1, prob.n)
    xs = spla.spsolve(A.tocsc(), b)
    x, it, hist, st = oracle.mg_pcg(prob, b, rtol=1e-13)
    assert st == oracle.OK
    assert np.linalg.norm(x - xs) <= 1e-10 * np.linalg.norm(xs)
    assert hist[-1] < 1e-13 and hist[0] == 1.0


def test_mg_pcg_error_decreases_in_the_energy_norm():
    prob = problem(16, 16, 8, a_v=1e4)
    A = assemble_A(prob.ah.reshape(16, 16), prob.h, prob.a_v, prob.mass)
    b = RNG.uniform(-1, 1, prob.n)
    xs = spla.spsolve(A.tocsc(), b)
    errs = []
    for k in range(1, 8):
        x, it, _, _ = oracle.mg_pcg(prob, b, rtol=0.0, maxit=k)
        assert it == k
        e = x - xs
        errs.append(e @ (A @ e))
    assert all(e1 < e0 for e0, e1 in zip(errs, errs[1:]))


def test_mg_pcg_needs_fewer_iterations_than_line_pcg():
    nx, ny, nz = 32, 32, 32
    h = W.layer_thickness(nz, True)
    ah = W.horizontal_coefficient(nx, ny, True)
    prob = oracle.Problem(nx, ny, nz, ah=ah, a_v=1e5, mass=1.0, h=h)
    b = W.uniform_rhs(prob.n, 3)
    x1, it1, _, st1 = oracle.pcg(prob, b, rtol=1e-10)
    x2, it2, _, st2 = oracle.mg_pcg(prob, b, rtol=1e-10)
    assert st1 == st2 == oracle.OK
    assert it2 * 2 < it1
    assert np.linalg.norm(x2 - x1) <= 1e-8 * np.linalg.norm(x1)
