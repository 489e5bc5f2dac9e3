"""A grid of more than 2^31 cells: 64-bit indexing everywhere on the path.

4096 x 4096 x 130 = 2,181,038,080 cells (17.4 GB per vector).  apply_A and
precond on the caller's layout are compared with the oracle on sampled cells
and columns: around linear index 2^31, at the end of the grid and at random;
then one PCG iteration from x0 = 0 must give x1 = alpha_0 M^{-1} b on every
cell, with alpha_0 = <b, z0> / <z0, A z0> formed from those two operators.
About 140 GB of device memory and 20 GB of host memory; skipped where less is
free.
"""
import os

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
NX, NY, NZ = 4096, 4096, 130
N = NX * NY * NZ
NEED_DEVICE = 170e9
NEED_HOST = 40e9


def host_free_bytes():
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def dot(a, b, chunk=1 << 30):
    # torch.dot's library call takes a 32-bit length
    return sum(float(torch.dot(a[i:i + chunk], b[i:i + chunk])) for i in range(0, a.numel(), chunk))


def test_grid_past_2_31_cells():
    assert N > 2 ** 31
    free, _ = torch.cuda.mem_get_info(DEV)
    if free < NEED_DEVICE:
        pytest.skip("%.0f GB of device memory free, %.0f needed" % (free / 1e9, NEED_DEVICE / 1e9))
    if host_free_bytes() < NEED_HOST:
        pytest.skip("not enough free host memory")
    h = W.layer_thickness(NZ, True)
    a_v = 1e4
    prob = oracle.Problem(NX, NY, NZ, ah=1.0, a_v=a_v, mass=1.0, h=h)
    b = np.random.default_rng(7).uniform(-1.0, 1.0, N)
    rng = np.random.default_rng(8)
    # cells: around 2^31, the last ones, random; columns holding them
    cells = np.concatenate([np.arange(2 ** 31 - 700, 2 ** 31 + 700), np.arange(N - 700, N),
                            rng.integers(0, N, 2000)]).astype(np.int64)
    cols = np.unique(np.concatenate([cells // NZ, [N // NZ - 1],
                                     rng.integers(0, NX * NY, 100)])).astype(np.int64)
    with mf.Solver(NX, NY, NZ, a_h=1.0, a_v=a_v, mass=1.0, dz=h) as s:
        bd = torch.from_numpy(b).to(DEV)
        y = torch.empty_like(bd)
        s.apply_A(bd, y)
        cd = torch.from_numpy(cells).to(DEV)
        got = y[cd].cpu().numpy()
        ref = oracle.apply_A_cells(prob, b, cells)
        assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
        s.precond(bd, y)                       # y = z0 = M^{-1} b
        colidx = (torch.from_numpy(cols).to(DEV)[:, None] * NZ +
                  torch.arange(NZ, device=DEV)[None, :])
        got = y[colidx].cpu().numpy()
        del colidx
        ref = oracle.precond_columns(prob, b, cols)
        assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
        x = torch.empty_like(bd)
        s.apply_A(y, x)                        # x = A z0
        alpha0 = dot(bd, y) / dot(y, x)
        assert alpha0 > 0.0
        x.zero_()
        it, hist, st = s.solve(bd, x, rtol=0.0, maxit=1)
        assert (it, st) == (1, mf.PCG_OK)
        assert np.all(np.isfinite(hist)) and hist[1] > 0.0
        # x1 - alpha0 z0 on every cell, in place
        zmax = max(float(y.max()), -float(y.min()))
        x.sub_(y, alpha=alpha0)
        err = float(x.abs_().max())
        assert err <= 1e-10 * alpha0 * zmax, (err, alpha0 * zmax)
    del bd, y, x
    torch.cuda.empty_cache()
