/*
 * oracle_pcg.c -- the CPU oracle for the matrix-free PCG solver.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, sequential, fp64 C, compiled with
 * -O2 -ffp-contract=off so every product and sum is rounded exactly as
 * written.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load it.  It shares no code, header or table with the
 * CUDA path.
 *
 * Source: E. Mueller, X. Guo, R. Scheichl, S. Shi, "Matrix-free GPU
 * implementation of a preconditioned conjugate gradient solver for
 * anisotropic elliptic PDEs" (2013).
 *
 * Grid and layout.  Cell (i,j,k) of an nx x ny x nz grid, i,j horizontal
 * (periodic), k vertical (0 = bottom), is stored at
 *     l = ((j*nx) + i)*nz + k,
 * i.e. every vertical column is contiguous (the column-major ordering of
 * section 3, eq. (10), and the CPU layout eq. (20)).
 *
 * Operator (section 3, eqs. (5)-(8); matrix-free stencil eq. (18)).  With
 * horizontal cell area |T| = 1 and unit horizontal spacing:
 *   d_k         = h_k                               (layer thickness)
 *   a_k         = mass * h_k                        (zero-order term)
 *   b_k         = -a_v / (0.5*(h_k + h_{k+1}))      (k < nz-1, else 0)
 *   c_k         = -a_v / (0.5*(h_{k-1} + h_k))      (k > 0,    else 0)
 *   alpha_{T,T'} = -0.5*(a_h(T) + a_h(T'))          (each horizontal face)
 *   alpha_T     = sum over the 4 faces of alpha_{T,T'}          (eq. (7))
 *   diagonal    = (a_k - b_k - c_k) - alpha_T * d_k              (eq. (8))
 *   (A u)_{T,k} = diagonal*u_{T,k} + b_k u_{T,k+1} + c_k u_{T,k-1}
 *                 + sum_{T'} alpha_{T,T'} d_k u_{T',k}           (eqs. (5),(6))
 * The off-diagonal entries b, c, alpha are the signed (negative) matrix
 * entries, which makes A symmetric positive definite.  A zero b_k / c_k at
 * the top / bottom is the homogeneous Neumann condition (no flux through
 * the lid or the floor).
 *
 * Preconditioner (section 4.1; eq. (19)).  M = blockdiag(A_T): the
 * horizontal couplings between columns are dropped, the diagonal keeps
 * alpha_T.  Each column's tridiagonal system is solved by the Thomas
 * algorithm (Gaussian elimination without pivoting for a tridiagonal matrix).
 *
 * Solver (section 4, left-preconditioned conjugate gradients, Hestenes and
 * Stiefel).  Textbook PCG; the stopping test ||r_k|| / ||r_0|| < rtol of
 * Algorithm 1 (tau = 0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK        0
#define ORACLE_EINVAL    1
#define ORACLE_ENOMEM    2
#define ORACLE_ENOTCONV  4
#define ORACLE_EBREAKDOWN 5

typedef struct {
  int nx, ny, nz;
  const double* ah;   /* horizontal coefficient a_h(i,j), nx*ny, index j*nx+i */
  double a_v;         /* vertical coefficient */
  double mass;        /* zero-order coefficient */
  const double* h;    /* layer thicknesses h_k, nz */
} grid_t;

static int check_grid(const grid_t* g) {
  if (g->nx < 1 || g->ny < 1 || g->nz < 1) return ORACLE_EINVAL;
  if (!g->ah || !g->h) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Vertical matrix entries of row k (eq. (8) with |T| = 1). */
static double entry_a(const grid_t* g, int k) { return g->mass * g->h[k]; }
static double entry_b(const grid_t* g, int k) {  /* coupling to k+1 */
  if (k >= g->nz - 1) return 0.0;
  return -g->a_v / (0.5 * (g->h[k] + g->h[k + 1]));
}
static double entry_c(const grid_t* g, int k) {  /* coupling to k-1 */
  if (k <= 0) return 0.0;
  return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k]));
}
static double entry_d(const grid_t* g, int k) { return g->h[k]; }

/* Horizontal neighbours of column (i,j), periodic in i and j. */
typedef struct { int64_t e, w, n, s; double ae, aw, an, as; } nbrs_t;

static nbrs_t neighbours(const grid_t* g, int i, int j) {
  nbrs_t nb;
  int ip = (i + 1) % g->nx, im = (i - 1 + g->nx) % g->nx;
  int jp = (j + 1) % g->ny, jm = (j - 1 + g->ny) % g->ny;
  int64_t c = (int64_t)j * g->nx + i;
  nb.e = (int64_t)j * g->nx + ip;
  nb.w = (int64_t)j * g->nx + im;
  nb.n = (int64_t)jp * g->nx + i;
  nb.s = (int64_t)jm * g->nx + i;
  /* alpha_{T,T'}: minus the face value of a_h, the mean of the two cells */
  nb.ae = -0.5 * (g->ah[c] + g->ah[nb.e]);
  nb.aw = -0.5 * (g->ah[c] + g->ah[nb.w]);
  nb.an = -0.5 * (g->ah[c] + g->ah[nb.n]);
  nb.as = -0.5 * (g->ah[c] + g->ah[nb.s]);
  return nb;
}

/* Row (i,j,k) of A applied to x. */
static double apply_row(const grid_t* g, int i, int j, int k, const double* x) {
  nbrs_t nb = neighbours(g, i, j);
  int64_t nz = g->nz;
  int64_t col = (int64_t)j * g->nx + i;
  int64_t l = col * nz + k;
  double alpha_T = nb.ae + nb.aw + nb.an + nb.as;          /* eq. (7) */
  double a = entry_a(g, k), b = entry_b(g, k), c = entry_c(g, k), d = entry_d(g, k);
  double diag = (a - b - c) - alpha_T * d;                  /* eq. (8) */
  double y = diag * x[l];
  if (k < g->nz - 1) y += b * x[l + 1];
  if (k > 0) y += c * x[l - 1];
  y += nb.ae * d * x[nb.e * nz + k];                        /* eq. (6) */
  y += nb.aw * d * x[nb.w * nz + k];
  y += nb.an * d * x[nb.n * nz + k];
  y += nb.as * d * x[nb.s * nz + k];
  return y;
}

static void apply_A(const grid_t* g, const double* x, double* y) {
  for (int j = 0; j < g->ny; ++j)
    for (int i = 0; i < g->nx; ++i)
      for (int k = 0; k < g->nz; ++k)
        y[((int64_t)j * g->nx + i) * g->nz + k] = apply_row(g, i, j, k, x);
}

/* Thomas algorithm for column (i,j) of M z = r (eq. (19)).  phi and y are
 * scratch of length nz.  Returns ORACLE_EBREAKDOWN if a pivot is not
 * positive (the column matrix is then not SPD). */
static int thomas_column(const grid_t* g, int i, int j, const double* r, double* z,
                         double* phi, double* y) {
  nbrs_t nb = neighbours(g, i, j);
  double alpha_T = nb.ae + nb.aw + nb.an + nb.as;
  int nz = g->nz;
  /* forward elimination */
  for (int k = 0; k < nz; ++k) {
    double a = entry_a(g, k), b = entry_b(g, k), c = entry_c(g, k), d = entry_d(g, k);
    double diag = (a - b - c) - alpha_T * d;
    double sub = c, sup = b;
    double D = (k == 0) ? diag : diag - sub * phi[k - 1];
    if (!(D > 0.0)) return ORACLE_EBREAKDOWN;
    phi[k] = sup / D;
    y[k] = (k == 0) ? r[k] / D : (r[k] - sub * y[k - 1]) / D;
  }
  /* back substitution */
  z[nz - 1] = y[nz - 1];
  for (int k = nz - 2; k >= 0; --k) z[k] = y[k] - phi[k] * z[k + 1];
  return ORACLE_OK;
}

static int precond(const grid_t* g, const double* r, double* z, double* phi, double* y) {
  for (int j = 0; j < g->ny; ++j)
    for (int i = 0; i < g->nx; ++i) {
      int64_t off = ((int64_t)j * g->nx + i) * g->nz;
      int st = thomas_column(g, i, j, r + off, z + off, phi, y);
      if (st) return st;
    }
  return ORACLE_OK;
}

static double dot(int64_t n, const double* a, const double* b) {
  double s = 0.0;
  for (int64_t l = 0; l < n; ++l) s += a[l] * b[l];
  return s;
}

/* ------------------------------------------------------------------ API */

int oracle_apply_A(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                   const double* h, const double* x, double* y) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h};
  if (check_grid(&g) || !x || !y) return ORACLE_EINVAL;
  apply_A(&g, x, y);
  return ORACLE_OK;
}

/* y at the listed linear cell indices only (for sampled checks of big grids). */
int oracle_apply_A_cells(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                         const double* h, const double* x, const int64_t* cells,
                         int64_t ncells, double* out) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h};
  if (check_grid(&g) || !x || (!cells && ncells) || (!out && ncells)) return ORACLE_EINVAL;
  int64_t n = (int64_t)nx * ny * nz;
  for (int64_t s = 0; s < ncells; ++s) {
    int64_t l = cells[s];
    if (l < 0 || l >= n) return ORACLE_EINVAL;
    int k = (int)(l % nz);
    int64_t col = l / nz;
    out[s] = apply_row(&g, (int)(col % nx), (int)(col / nx), k, x);
  }
  return ORACLE_OK;
}

int oracle_precond(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                   const double* h, const double* r, double* z) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h};
  if (check_grid(&g) || !r || !z) return ORACLE_EINVAL;
  double* phi = (double*)malloc(sizeof(double) * nz);
  double* y = (double*)malloc(sizeof(double) * nz);
  if (!phi || !y) { free(phi); free(y); return ORACLE_ENOMEM; }
  int st = precond(&g, r, z, phi, y);
  free(phi); free(y);
  return st;
}

/* z = M^{-1} r for the listed columns (index j*nx+i) only; zcols is
 * ncols*nz, one column after another. */
int oracle_precond_columns(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                           const double* h, const double* r, const int64_t* cols,
                           int64_t ncols, double* zcols) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h};
  if (check_grid(&g) || !r || (!cols && ncols) || (!zcols && ncols)) return ORACLE_EINVAL;
  double* phi = (double*)malloc(sizeof(double) * nz);
  double* y = (double*)malloc(sizeof(double) * nz);
  if (!phi || !y) { free(phi); free(y); return ORACLE_ENOMEM; }
  int st = ORACLE_OK;
  for (int64_t s = 0; s < ncols && !st; ++s) {
    int64_t col = cols[s];
    if (col < 0 || col >= (int64_t)nx * ny) { st = ORACLE_EINVAL; break; }
    st = thomas_column(&g, (int)(col % nx), (int)(col / nx), r + col * nz,
                       zcols + s * nz, phi, y);
  }
  free(phi); free(y);
  return st;
}

/* Textbook left-preconditioned CG.  x holds x_0 on entry and the final
 * iterate on return.  hist (maxit+1 entries, or NULL) receives
 * ||r_k|| / ||r_0|| for k = 0..iters.  The stopping test is the one of
 * Algorithm 1 with tau = 0: stop at the first k with ||r_k||/||r_0|| < rtol;
 * an exactly zero residual also stops.  rtol = 0 runs exactly maxit
 * iterations.  *iters is the number of products A p performed. */
int oracle_pcg(int nx, int ny, int nz, const double* ah, double a_v, double mass,
               const double* h, const double* b, double* x, double rtol, int maxit,
               int* iters, double* hist) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h};
  if (check_grid(&g) || !b || !x || !iters || maxit < 0 || !(rtol >= 0.0)) return ORACLE_EINVAL;
  int64_t n = (int64_t)nx * ny * nz;
  double* r = (double*)malloc(sizeof(double) * n);
  double* z = (double*)malloc(sizeof(double) * n);
  double* p = (double*)malloc(sizeof(double) * n);
  double* q = (double*)malloc(sizeof(double) * n);
  double* phi = (double*)malloc(sizeof(double) * nz);
  double* yv = (double*)malloc(sizeof(double) * nz);
  int st = ORACLE_OK;
  if (!r || !z || !p || !q || !phi || !yv) { st = ORACLE_ENOMEM; goto done; }

  /* r_0 = b - A x_0,  z_0 = M^{-1} r_0,  p_0 = z_0 */
  apply_A(&g, x, q);
  for (int64_t l = 0; l < n; ++l) r[l] = b[l] - q[l];
  double rho0 = sqrt(dot(n, r, r));
  *iters = 0;
  if (hist) hist[0] = (rho0 > 0.0) ? 1.0 : 0.0;
  if (rho0 == 0.0) goto done;
  if (!(rho0 < INFINITY)) { st = ORACLE_EBREAKDOWN; goto done; }
  if (1.0 < rtol) goto done;
  st = precond(&g, r, z, phi, yv);
  if (st) goto done;
  memcpy(p, z, sizeof(double) * n);
  double kappa = dot(n, r, z);
  if (!(kappa > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }

  for (int k = 1; k <= maxit; ++k) {
    apply_A(&g, p, q);                          /* q = A p */
    double sigma = dot(n, p, q);
    if (!(sigma > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }
    double alpha = kappa / sigma;
    for (int64_t l = 0; l < n; ++l) x[l] += alpha * p[l];
    for (int64_t l = 0; l < n; ++l) r[l] -= alpha * q[l];
    double rnorm = sqrt(dot(n, r, r));
    double res = rnorm / rho0;
    if (hist) hist[k] = res;
    *iters = k;
    if (res < rtol || rnorm == 0.0) goto done;
    if (!(res < INFINITY)) { st = ORACLE_EBREAKDOWN; goto done; }
    if (k == maxit) break;
    st = precond(&g, r, z, phi, yv);            /* z = M^{-1} r */
    if (st) goto done;
    double kappa_new = dot(n, r, z);
    if (!(kappa_new > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }
    double beta = kappa_new / kappa;
    kappa = kappa_new;
    for (int64_t l = 0; l < n; ++l) p[l] = z[l] + beta * p[l];
  }
  if (rtol > 0.0) st = ORACLE_ENOTCONV;
done:
  free(r); free(z); free(p); free(q); free(phi); free(yv);
  return st;
}
