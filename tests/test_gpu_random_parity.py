"""Seeded random cases, GPU vs the CPU oracle.

Grid sizes across tile boundaries and the tensor-memory heights, a_h fields
with jumps (log-normal per column), random layer thicknesses, vertical
coefficients and mass terms over several decades: apply_A and precond to
1e-12 relative max-norm, and solves to a 1e-10 residual in three solver
modes (iteration count within one of the oracle's, the iterate at the
oracle's count within 1e-8).  The generator draws every case from one seed,
so a failure names a reproducible case.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import matrix_free_pcg_gb300 as mf  # noqa: E402

DEV = torch.device("cuda:0")
NZ_CHOICES = [1, 2, 3, 5, 8, 16, 31, 32, 33, 48, 64, 100, 128, 129, 200]


def draw(i):
    """Case i: (nx, ny, nz, a_h field or None, a_h, a_v, mass, h, seed)."""
    g = np.random.default_rng(1000 + i)
    nx = int(g.integers(1, 97))
    ny = int(g.integers(1, 71))
    nz = int(g.choice(NZ_CHOICES))
    if g.random() < 0.6:
        ah = np.exp(g.normal(0.0, 0.7, size=(ny, nx)))   # jumps from column to column
        a_h = 1.0
    else:
        ah, a_h = None, float(np.exp(g.normal(0.0, 0.7)))
    a_v = float(10.0 ** g.uniform(0.0, 5.0))
    mass = float(10.0 ** g.uniform(-2.0, 1.0))
    if g.random() < 0.5:
        h = g.uniform(0.5, 2.0, size=nz)                 # irregular layers
    else:
        q = g.uniform(1.0, 1.08)
        h = q ** np.arange(nz, dtype=np.float64)         # graded layers
        h *= nz / h.sum()
    return nx, ny, nz, ah, a_h, a_v, mass, h, 2000 + i


CASES = list(range(24))


def problem(i):
    nx, ny, nz, ah, a_h, a_v, mass, h, seed = draw(i)
    prob = oracle.Problem(nx, ny, nz, ah=ah if ah is not None else a_h, a_v=a_v, mass=mass, h=h)
    kw = dict(a_h=a_h, a_h_field=ah, a_v=a_v, mass=mass, dz=h)
    b = np.random.default_rng(seed).uniform(-1.0, 1.0, nx * ny * nz)
    return prob, kw, b


def rel_maxdiff(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("i", CASES)
def test_random_operators_match_oracle(i):
    prob, kw, x = problem(i)
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        xd = torch.from_numpy(x).to(DEV)
        y = s.apply_A(xd).cpu().numpy()
        z = s.precond(xd).cpu().numpy()
    assert rel_maxdiff(y, oracle.apply_A(prob, x)) <= 1e-12, draw(i)[:3]
    assert rel_maxdiff(z, oracle.precond(prob, x)) <= 1e-12, draw(i)[:3]


@pytest.mark.parametrize("mode", ["tiled", "column", "persistent"])
@pytest.mark.parametrize("i", CASES)
def test_random_solves_match_oracle(i, mode):
    prob, kw, b = problem(i)
    x_ref, it_ref, _, st_ref = oracle.pcg(prob, b, rtol=1e-10, maxit=1000)
    assert st_ref == oracle.OK
    with mf.Solver(prob.nx, prob.ny, prob.nz, **kw) as s:
        if mode == "column":
            s.set_layout("column")
        elif mode == "persistent":
            s.set_loop("persistent")
        bd = torch.from_numpy(b).to(DEV)
        x = torch.zeros_like(bd)
        it, hist, st = s.solve(bd, x, rtol=1e-10, maxit=1000)
        assert st == mf.PCG_OK and abs(it - it_ref) <= 1, (draw(i)[:3], it, it_ref)
        x.zero_()
        it2, _, st2 = s.solve(bd, x, rtol=0.0, maxit=it_ref)
        assert (it2, st2) == (it_ref, mf.PCG_OK)
        xs = x.cpu().numpy()
    assert np.linalg.norm(xs - x_ref) <= 1e-8 * np.linalg.norm(x_ref), draw(i)[:3]
