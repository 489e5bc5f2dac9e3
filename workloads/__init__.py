"""Seeded synthetic workloads for the anisotropic elliptic PCG solve.

This module holds the input generators only: grid sizes, the coefficient
data (layer thicknesses, the horizontal coefficient field) and right-hand
sides, all drawn with numpy's PCG64 generator in the memory order of the
column-contiguous layout (numpy shape (ny, nx, nz), C order; linear index
((j*nx)+i)*nz + k).  It contains none of the solver's arithmetic, so both
the CUDA path and the CPU oracle may use it.

The five workloads are flat 3D grids with a strong vertical anisotropy, the
setting of Mueller et al., "Matrix-free GPU implementation of a
preconditioned conjugate gradient solver for anisotropic elliptic PDEs"
(section 3: a tensor-product grid with a graded vertical spacing, n_z of
order 100).
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    nx: int
    ny: int
    nz: int
    a_v: float             # vertical coefficient
    a_h: float = 1.0       # horizontal coefficient (its mean when varying)
    varying_ah: bool = False
    graded: bool = False   # geometric layer thicknesses, ratio 1.05 per level
    mass: float = 1.0
    rhs: str = "uniform"   # "uniform" | "manufactured" | "bumps"
    seed: int = 0
    rtol: float = 1e-10
    maxit: int = 500       # with rtol == 0 exactly maxit iterations are run

    @property
    def n(self):
        return self.nx * self.ny * self.nz

    @property
    def shape(self):
        return (self.ny, self.nx, self.nz)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("aniso_32x32x16", 32, 32, 16, a_v=100.0, rhs="uniform", seed=0,
                 rtol=1e-10, maxit=500),
        Workload("manufactured_128x128x64", 128, 128, 64, a_v=1e3, rhs="manufactured",
                 seed=1, rtol=1e-10, maxit=500),
        Workload("graded_512x512x64", 512, 512, 64, a_v=1e4, graded=True, rhs="uniform",
                 seed=2, rtol=1e-10, maxit=500),
        Workload("graded_varcoef_1024x1024x128", 1024, 1024, 128, a_v=1e5, graded=True,
                 varying_ah=True, rhs="uniform", seed=3, rtol=1e-10, maxit=500),
        Workload("bumps_2048x2048x64", 2048, 2048, 64, a_v=1e4, rhs="bumps", seed=4,
                 rtol=0.0, maxit=50),
    ]
}
HEADLINE = "graded_varcoef_1024x1024x128"


def layer_thickness(nz, graded):
    """Layer thicknesses h_k, k = 0 (bottom) .. nz-1.

    Uniform: all ones.  Graded: h_k proportional to 1.05**k (finest at the
    bottom), scaled so that the mean thickness is 1.
    """
    if not graded:
        return np.ones(nz)
    g = 1.05 ** np.arange(nz, dtype=np.float64)
    return g * (nz / g.sum())


def horizontal_coefficient(nx, ny, varying, a_h=1.0):
    """a_h(i,j) as an (ny, nx) array (row j, column i).

    Varying: a_h(i,j) = 1 + 0.5*sin(2*pi*i/nx)*cos(2*pi*j/ny).
    """
    if not varying:
        return np.full((ny, nx), float(a_h))
    i = np.arange(nx, dtype=np.float64)
    j = np.arange(ny, dtype=np.float64)
    return 1.0 + 0.5 * np.outer(np.cos(2.0 * np.pi * j / ny), np.sin(2.0 * np.pi * i / nx))


def uniform_rhs(n, seed):
    return np.random.default_rng(seed).uniform(-1.0, 1.0, n)


def manufactured_solution(n, seed):
    """u* ~ N(0,1) i.i.d.; the right-hand side is then A u*."""
    return np.random.default_rng(seed).standard_normal(n)


def gaussian_bumps(nx, ny, nz, seed, nbumps=16):
    """Sum of nbumps unit-amplitude Gaussian bumps, shape (ny, nx, nz).

    Bump b: centre (i_b, j_b, k_b) ~ U[0,nx) x U[0,ny) x U[0,nz), width
    w_b ~ U[5, 50) cells, drawn in that order bump after bump.  The distance
    between cell centres is the minimum periodic image in i and j and plain in
    k; exp(-d^2/(2 w^2)) is evaluated as the product of its three 1-D factors.
    """
    rng = np.random.default_rng(seed)
    params = []
    for _ in range(nbumps):
        ic = rng.uniform(0, nx)
        jc = rng.uniform(0, ny)
        kc = rng.uniform(0, nz)
        w = rng.uniform(5, 50)
        params.append((ic, jc, kc, w))

    def wrap(d, period):
        return (d + 0.5 * period) % period - 0.5 * period

    out = np.zeros((ny, nx, nz))
    ci = np.arange(nx) + 0.5
    cj = np.arange(ny) + 0.5
    ck = np.arange(nz) + 0.5
    for ic, jc, kc, w in params:
        gi = np.exp(-wrap(ci - ic, nx) ** 2 / (2 * w * w))
        gj = np.exp(-wrap(cj - jc, ny) ** 2 / (2 * w * w))
        gk = np.exp(-((ck - kc) ** 2) / (2 * w * w))
        gik = np.outer(gi, gk)                      # (nx, nz)
        for j0 in range(0, ny, 256):                # bounded temporaries
            j1 = min(ny, j0 + 256)
            out[j0:j1] += gj[j0:j1, None, None] * gik[None, :, :]
    return out


def make_inputs(w):
    """(h, ah, vec) for a workload.  vec is the right-hand side, except for
    the manufactured workload where it is u* (b = A u* is formed by the
    caller with its own operator)."""
    h = layer_thickness(w.nz, w.graded)
    ah = horizontal_coefficient(w.nx, w.ny, w.varying_ah, w.a_h)
    if w.rhs == "uniform":
        vec = uniform_rhs(w.n, w.seed)
    elif w.rhs == "manufactured":
        vec = manufactured_solution(w.n, w.seed)
    elif w.rhs == "bumps":
        vec = gaussian_bumps(w.nx, w.ny, w.nz, w.seed).reshape(-1)
    else:
        raise ValueError(w.rhs)
    return h, ah, vec
