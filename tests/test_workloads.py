"""The seeded input generators against their stated recipes: graded layers
with ratio 1.05 per level and mean thickness 1 (closed form of the geometric
sum), the varying a_h field's range and mean, and the Gaussian bumps'
bounds, periodic wrap and seeding."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("nz", [1, 16, 64, 128])
def test_graded_layers_are_geometric_with_mean_one(nz):
    h = W.layer_thickness(nz, graded=True)
    assert h.shape == (nz,) and np.all(h > 0)
    assert abs(h.mean() - 1.0) <= 1e-14
    if nz > 1:
        np.testing.assert_allclose(h[1:] / h[:-1], 1.05, rtol=1e-14)
    # h_0 = nz (r - 1) / (r^nz - 1): the geometric sum in closed form
    h0 = nz * 0.05 / (1.05 ** nz - 1.0) if nz > 1 else 1.0
    assert abs(h[0] - h0) <= 1e-14 * h0
    assert np.array_equal(W.layer_thickness(nz, graded=False), np.ones(nz))


def test_graded_layer_extremes_at_the_workload_depths():
    h64, h128 = W.layer_thickness(64, True), W.layer_thickness(128, True)
    assert (round(h64[0], 4), round(h64[-1], 3)) == (0.1474, 3.188)
    assert (round(h128[0], 5), round(h128[-1], 3)) == (0.01244, 6.107)


@pytest.mark.parametrize("shape", [(16, 12), (1024, 1024), (5, 3)])
def test_varying_coefficient_field(shape):
    nx, ny = shape
    ah = W.horizontal_coefficient(nx, ny, varying=True)
    assert ah.shape == (ny, nx)
    assert ah.min() >= 0.5 - 1e-15 and ah.max() <= 1.5 + 1e-15
    # a full period of sin in i: the mean over i is 1 for every j
    np.testing.assert_allclose(ah.mean(axis=1), 1.0, atol=1e-14)
    i, j = 3 % nx, 2 % ny
    want = 1.0 + 0.5 * np.sin(2 * np.pi * i / nx) * np.cos(2 * np.pi * j / ny)
    assert abs(ah[j, i] - want) <= 1e-15
    assert np.array_equal(W.horizontal_coefficient(nx, ny, False, 0.7), np.full((ny, nx), 0.7))


def test_bumps_bounds_wrap_and_seed():
    nx, ny, nz = 64, 48, 16
    f = W.gaussian_bumps(nx, ny, nz, seed=9, nbumps=4)
    assert f.shape == (ny, nx, nz) and np.all(f > 0) and f.max() <= 4.0
    assert np.array_equal(f, W.gaussian_bumps(nx, ny, nz, seed=9, nbumps=4))
    assert not np.array_equal(f, W.gaussian_bumps(nx, ny, nz, seed=10, nbumps=4))
    # one bump: periodic in i and j, so the cells at the same periodic
    # distance on either side of its centre hold the same value
    g = W.gaussian_bumps(nx, ny, nz, seed=3, nbumps=1)
    rng = np.random.default_rng(3)
    ic, jc = rng.uniform(0, nx), rng.uniform(0, ny)
    di = ((np.arange(nx) + 0.5 - ic + nx / 2) % nx) - nx / 2
    dj = ((np.arange(ny) + 0.5 - jc + ny / 2) % ny) - ny / 2
    # the profile along i (any j, k) decreases with the periodic distance
    row = g[0, :, 0]
    order = np.argsort(np.abs(di))
    assert np.all(np.diff(row[order]) <= 1e-15)
    col = g[:, 0, 0]
    assert np.all(np.diff(col[np.argsort(np.abs(dj))]) <= 1e-15)


def test_workloads_are_seeded_and_sized():
    # inputs drawn for the grids small enough for a CPU test (up to 4 M cells)
    for w in W.WORKLOADS.values():
        assert w.n == w.nx * w.ny * w.nz
        if w.n <= 1 << 22:
            h, ah, vec = W.make_inputs(w)
            assert h.shape == (w.nz,) and ah.shape == (w.ny, w.nx) and vec.size == w.n
            assert np.array_equal(vec, W.make_inputs(w)[2])
    assert W.HEADLINE in W.WORKLOADS
