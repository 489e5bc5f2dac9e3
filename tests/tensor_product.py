"""Independent constructions used to pin the oracle (tests only).

The operator is assembled here from the tensor-product form of section 3,
eq. (3), of Mueller et al. ("Matrix-free GPU implementation of a
preconditioned conjugate gradient solver for anisotropic elliptic PDEs"):

    A = D_h (x) diag(h)  +  I_h (x) D_v  +  mass * I_h (x) diag(h)

with D_h the periodic horizontal graph Laplacian whose face weights are the
mean of a_h over the two cells, and D_v the vertical Neumann Laplacian with
face transmissibilities a_v / (0.5*(h_k + h_{k+1})).  Nothing here is
shared with the oracle's stencil code: the matrices come from face lists and
Kronecker products, not from eq. (18).
"""
import numpy as np
import scipy.sparse as sp


def horizontal_laplacian(ah):
    """Periodic graph Laplacian on an (ny, nx) grid, one entry per face."""
    ny, nx = ah.shape
    n = nx * ny
    rows, cols, vals = [], [], []

    def add_face(c1, c2, w):
        rows.extend([c1, c2, c1, c2])
        cols.extend([c1, c2, c2, c1])
        vals.extend([w, w, -w, -w])

    for j in range(ny):
        for i in range(nx):
            c = j * nx + i
            e = j * nx + (i + 1) % nx
            nn = ((j + 1) % ny) * nx + i
            add_face(c, e, 0.5 * (ah[j, i] + ah[j, (i + 1) % nx]))
            add_face(c, nn, 0.5 * (ah[j, i] + ah[(j + 1) % ny, i]))
    return sp.csr_matrix((vals, (rows, cols)), shape=(n, n))


def face_sums(ah):
    """sum of the four face weights of every column (alpha_T up to sign)."""
    ny, nx = ah.shape
    s = np.zeros(nx * ny)
    for j in range(ny):
        for i in range(nx):
            a = ah[j, i]
            s[j * nx + i] = 0.5 * (4 * a + ah[j, (i + 1) % nx] + ah[j, (i - 1) % nx]
                                   + ah[(j + 1) % ny, i] + ah[(j - 1) % ny, i])
    return s


def vertical_laplacian(h, a_v):
    nz = len(h)
    t = a_v / (0.5 * (h[:-1] + h[1:]))          # nz-1 interior faces
    main = np.zeros(nz)
    main[:-1] += t
    main[1:] += t
    return sp.diags([main, -t, -t], [0, 1, -1], shape=(nz, nz), format="csr")


def assemble_A(ah, h, a_v, mass, area=1.0):
    """The operator on cells of horizontal area `area` (square cells): the
    horizontal face weights keep their form, the vertical and zero-order
    terms are integrated over the larger cells."""
    ny, nx = ah.shape
    Dh = horizontal_laplacian(ah)
    Dv = vertical_laplacian(h, a_v)
    H = sp.diags(h)
    I = sp.identity(nx * ny, format="csr")
    return (sp.kron(Dh, H) + area * (sp.kron(I, Dv) + mass * sp.kron(I, H))).tocsr()


def assemble_M(ah, h, a_v, mass, area=1.0):
    """Column preconditioner of eq. (19): per column, the vertical operator
    plus the horizontal diagonal sum(a_f) h_k plus the mass term."""
    ny, nx = ah.shape
    Dv = vertical_laplacian(h, a_v)
    H = sp.diags(h)
    I = sp.identity(nx * ny, format="csr")
    S = sp.diags(face_sums(ah))
    return (sp.kron(S, H) + area * (sp.kron(I, Dv) + mass * sp.kron(I, H))).tocsr()


def piecewise_constant_prolongation(nx, ny, nz):
    """P: (nx*ny*nz) x (nx/2*ny/2*nz) 0/1 matrix, fine cell (i,j,k) <- coarse
    cell (i//2, j//2, k), built from index maps."""
    rows, cols = [], []
    for j in range(ny):
        for i in range(nx):
            for k in range(nz):
                rows.append((j * nx + i) * nz + k)
                cols.append(((j // 2) * (nx // 2) + i // 2) * nz + k)
    return sp.csr_matrix((np.ones(len(rows)), (rows, cols)),
                         shape=(nx * ny * nz, (nx // 2) * (ny // 2) * nz))


def block_diagonal_part(A, nz):
    """Entries of A that couple cells of the same column only."""
    A = A.tocoo()
    keep = (A.row // nz) == (A.col // nz)
    return sp.csr_matrix((A.data[keep], (A.row[keep], A.col[keep])), shape=A.shape)


def fourier_mode(nx, ny, nz, p, q, m):
    """cos(2 pi (p i/nx + q j/ny)) cos(pi m (k+1/2)/nz) in the (ny, nx, nz) layout."""
    i = np.arange(nx)[None, :, None]
    j = np.arange(ny)[:, None, None]
    k = np.arange(nz)[None, None, :]
    return (np.cos(2 * np.pi * (p * i / nx + q * j / ny)) *
            np.cos(np.pi * m * (k + 0.5) / nz)).reshape(-1)
