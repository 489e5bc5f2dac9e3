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
 *
 * OpenMP.  The benchmark's second, labelled CPU line builds this same file
 * with -fopenmp (liboracle_pcg_omp.so): the loops over cells and columns of
 * the line-preconditioned PCG then run on all host cores, and the dot
 * products add per-thread partial sums.  That build is a timing baseline
 * only.  The sequential build, which the tests and every comparison with the
 * GPU use, does not see the OpenMP lines: its arithmetic and its order are
 * the ones written.
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

#ifdef _OPENMP
#define OMP_PRAGMA(x) _Pragma(#x)
#define OMP_FOR OMP_PRAGMA(omp parallel for schedule(static))
#define OMP_FOR_SUM(v) OMP_PRAGMA(omp parallel for schedule(static) reduction(+ : v))
#else
#define OMP_FOR
#define OMP_FOR_SUM(v)
#endif

typedef struct {
  int nx, ny, nz;
  const double* ah;   /* horizontal coefficient a_h(i,j), nx*ny, index j*nx+i */
  double a_v;         /* vertical coefficient */
  double mass;        /* zero-order coefficient */
  const double* h;    /* layer thicknesses h_k, nz */
  double area;        /* horizontal cell area |T| (1 on the given grid; 4^l on the
                         multigrid level l, whose cells are 2^l x 2^l columns) */
} grid_t;

static int check_grid(const grid_t* g) {
  if (g->nx < 1 || g->ny < 1 || g->nz < 1) return ORACLE_EINVAL;
  if (!g->ah || !g->h) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Vertical matrix entries of row k (eq. (8)): the zero-order and vertical
 * terms carry the horizontal cell area |T| (1 on the given grid, where these
 * are the entries with |T| = 1). */
static double entry_a(const grid_t* g, int k) { return g->mass * g->h[k] * g->area; }
static double entry_b(const grid_t* g, int k) {  /* coupling to k+1 */
  if (k >= g->nz - 1) return 0.0;
  return -g->a_v / (0.5 * (g->h[k] + g->h[k + 1])) * g->area;
}
static double entry_c(const grid_t* g, int k) {  /* coupling to k-1 */
  if (k <= 0) return 0.0;
  return -g->a_v / (0.5 * (g->h[k - 1] + g->h[k])) * g->area;
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
  OMP_FOR
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
#ifdef _OPENMP
  /* OpenMP build: the columns in parallel, each thread with its own scratch;
   * the status is that of any column that fails */
  int st = ORACLE_OK;
  const int64_t ncols = (int64_t)g->nx * g->ny;
  (void)phi;
  (void)y;
#pragma omp parallel reduction(max : st)
  {
    /* the thread's copy of st (a max reduction's starts at INT_MIN) */
    double* tphi = (double*)malloc(sizeof(double) * g->nz);
    double* ty = (double*)malloc(sizeof(double) * g->nz);
    st = (tphi && ty) ? ORACLE_OK : ORACLE_ENOMEM;
#pragma omp for schedule(static)
    for (int64_t c = 0; c < ncols; ++c) {
      if (st == ORACLE_OK) {
        int64_t off = c * g->nz;
        st = thomas_column(g, (int)(c % g->nx), (int)(c / g->nx), r + off, z + off, tphi, ty);
      }
    }
    free(tphi);
    free(ty);
  }
  return st;
#else
  for (int j = 0; j < g->ny; ++j)
    for (int i = 0; i < g->nx; ++i) {
      int64_t off = ((int64_t)j * g->nx + i) * g->nz;
      int st = thomas_column(g, i, j, r + off, z + off, phi, y);
      if (st) return st;
    }
  return ORACLE_OK;
#endif
}

static double dot(int64_t n, const double* a, const double* b) {
  double s = 0.0;
  OMP_FOR_SUM(s)
  for (int64_t l = 0; l < n; ++l) s += a[l] * b[l];
  return s;
}

/* ------------------------------------------------------------------ API */

int oracle_apply_A(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                   const double* h, const double* x, double* y) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
  if (check_grid(&g) || !x || !y) return ORACLE_EINVAL;
  apply_A(&g, x, y);
  return ORACLE_OK;
}

/* y at the listed linear cell indices only (for sampled checks of big grids). */
int oracle_apply_A_cells(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                         const double* h, const double* x, const int64_t* cells,
                         int64_t ncells, double* out) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
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
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
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
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
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

/* The preconditioner of the PCG loop: z = B r. */
typedef int (*prec_fn)(void* ctx, const double* r, double* z);

typedef struct { const grid_t* g; double* phi; double* y; } line_prec_t;

static int line_prec(void* c, const double* r, double* z) {
  line_prec_t* lp = (line_prec_t*)c;
  return precond(lp->g, r, z, lp->phi, lp->y);
}

/* Textbook left-preconditioned CG with the preconditioner `prec`.  x holds
 * x_0 on entry and the final iterate on return.  hist (maxit+1 entries, or
 * NULL) receives ||r_k|| / ||r_0|| for k = 0..iters.  The stopping test is
 * the one of Algorithm 1 with tau = 0: stop at the first k with
 * ||r_k||/||r_0|| < rtol; an exactly zero residual also stops.  rtol = 0 runs
 * exactly maxit iterations.  *iters is the number of products A p performed. */
static int pcg_loop(const grid_t* g, prec_fn prec, void* pctx, const double* b, double* x,
                    double rtol, int maxit, int* iters, double* hist) {
  int64_t n = (int64_t)g->nx * g->ny * g->nz;
  double* r = (double*)malloc(sizeof(double) * n);
  double* z = (double*)malloc(sizeof(double) * n);
  double* p = (double*)malloc(sizeof(double) * n);
  double* q = (double*)malloc(sizeof(double) * n);
  int st = ORACLE_OK;
  if (!r || !z || !p || !q) { st = ORACLE_ENOMEM; goto done; }

  /* r_0 = b - A x_0,  z_0 = B r_0,  p_0 = z_0 */
  apply_A(g, x, q);
  OMP_FOR
  for (int64_t l = 0; l < n; ++l) r[l] = b[l] - q[l];
  double rho0 = sqrt(dot(n, r, r));
  *iters = 0;
  if (hist) hist[0] = (rho0 > 0.0) ? 1.0 : 0.0;
  if (rho0 == 0.0) goto done;
  if (!(rho0 < INFINITY)) { st = ORACLE_EBREAKDOWN; goto done; }
  if (1.0 < rtol) goto done;
  st = prec(pctx, r, z);
  if (st) goto done;
  memcpy(p, z, sizeof(double) * n);
  double kappa = dot(n, r, z);
  if (!(kappa > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }

  for (int k = 1; k <= maxit; ++k) {
    apply_A(g, p, q);                           /* q = A p */
    double sigma = dot(n, p, q);
    if (!(sigma > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }
    double alpha = kappa / sigma;
    OMP_FOR
    for (int64_t l = 0; l < n; ++l) x[l] += alpha * p[l];
    OMP_FOR
    for (int64_t l = 0; l < n; ++l) r[l] -= alpha * q[l];
    double rnorm = sqrt(dot(n, r, r));
    double res = rnorm / rho0;
    if (hist) hist[k] = res;
    *iters = k;
    if (res < rtol || rnorm == 0.0) goto done;
    if (!(res < INFINITY)) { st = ORACLE_EBREAKDOWN; goto done; }
    if (k == maxit) break;
    st = prec(pctx, r, z);                      /* z = B r */
    if (st) goto done;
    double kappa_new = dot(n, r, z);
    if (!(kappa_new > 0.0)) { st = ORACLE_EBREAKDOWN; goto done; }
    double beta = kappa_new / kappa;
    kappa = kappa_new;
    OMP_FOR
    for (int64_t l = 0; l < n; ++l) p[l] = z[l] + beta * p[l];
  }
  if (rtol > 0.0) st = ORACLE_ENOTCONV;
done:
  free(r); free(z); free(p); free(q);
  return st;
}

/* PCG with the column preconditioner M of eq. (19). */
int oracle_pcg(int nx, int ny, int nz, const double* ah, double a_v, double mass,
               const double* h, const double* b, double* x, double rtol, int maxit,
               int* iters, double* hist) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
  if (check_grid(&g) || !b || !x || !iters || maxit < 0 || !(rtol >= 0.0)) return ORACLE_EINVAL;
  double* phi = (double*)malloc(sizeof(double) * nz);
  double* yv = (double*)malloc(sizeof(double) * nz);
  int st = ORACLE_ENOMEM;
  if (phi && yv) {
    line_prec_t lp = {&g, phi, yv};
    st = pcg_loop(&g, line_prec, &lp, b, x, rtol, maxit, iters, hist);
  }
  free(phi); free(yv);
  return st;
}

/* ------------------------------------------ tensor-product multigrid (V-cycle)
 *
 * The paper (sections 1, 2 and 9) names the column solve of eq. (19) as the
 * smoother of a geometric multigrid method built on the tensor-product idea
 * of Boerm and Hiptmair: the strong vertical coupling is handled exactly by
 * the line relaxation, so only the horizontal directions are coarsened.  The
 * pages leave the grid hierarchy, the intergrid operators and the cycle open;
 * the readings taken here are
 *   - levels: level l+1 merges the 2 x 2 columns (2I..2I+1, 2J..2J+1) of
 *     level l into column (I, J); all nz layers are kept.  Coarsening stops
 *     when nx or ny is odd (so a power-of-two grid goes down to one column)
 *     or when max_levels levels exist;
 *   - coarse operators by rediscretisation: level l is eqs. (5)-(8) on cells
 *     of horizontal area |T| = 4^l.  The horizontal face weight keeps its form
 *     (face length over centre distance is 1 on every level), its a_h being
 *     the mean of a_h over the 4 merged columns, level by level;
 *   - transfers: prolongation P copies a coarse column into its 4 fine
 *     columns (piecewise constant); restriction R = P^T sums the 4 fine
 *     values (the equations are integrated over the cells);
 *   - smoother: damped line relaxation x <- x + omega M_l^{-1} (b - A_l x)
 *     with the column preconditioner M_l of eq. (19) on level l;
 *   - cycle: from x = 0, nu smoothing steps, coarse-grid correction
 *     x <- x + P V_{l+1}(R (b - A_l x)), nu smoothing steps; on the coarsest
 *     level, nu smoothing steps from x = 0.  B = V_0 is symmetric, so it can
 *     precondition CG.
 */
#define ORACLE_MG_MAXLEV 32

typedef struct {
  int nlev;
  grid_t g[ORACLE_MG_MAXLEV];
  double* ah[ORACLE_MG_MAXLEV];                 /* coarse a_h (owned from level 1) */
  double *b[ORACLE_MG_MAXLEV], *x[ORACLE_MG_MAXLEV];
  double *t[ORACLE_MG_MAXLEV], *z[ORACLE_MG_MAXLEV];
  double *phi, *y;                              /* Thomas scratch, nz each */
  int nu;
  double omega;
} mg_t;

static int mg_count_levels(int nx, int ny, int max_levels) {
  int L = 1;
  while (L < ORACLE_MG_MAXLEV && (max_levels <= 0 || L < max_levels) && nx % 2 == 0 &&
         ny % 2 == 0) {
    nx /= 2;
    ny /= 2;
    ++L;
  }
  return L;
}

/* a_h of the coarse column (I, J): the mean over its 4 fine columns. */
static void mg_coarse_ah(int nxf, int nyf, const double* ahf, double* ahc) {
  int nxc = nxf / 2, nyc = nyf / 2;
  for (int J = 0; J < nyc; ++J)
    for (int I = 0; I < nxc; ++I) {
      double s = ahf[(2 * J) * nxf + 2 * I] + ahf[(2 * J) * nxf + 2 * I + 1] +
                 ahf[(2 * J + 1) * nxf + 2 * I] + ahf[(2 * J + 1) * nxf + 2 * I + 1];
      ahc[J * nxc + I] = 0.25 * s;
    }
}

/* r_c = R r_f: per layer, the sum of the 4 fine columns of each coarse one. */
static void mg_restrict(const grid_t* f, const double* rf, double* rc) {
  int nxc = f->nx / 2, nyc = f->ny / 2, nz = f->nz;
  for (int J = 0; J < nyc; ++J)
    for (int I = 0; I < nxc; ++I) {
      int64_t c00 = ((int64_t)(2 * J) * f->nx + 2 * I) * nz;
      int64_t c10 = ((int64_t)(2 * J) * f->nx + 2 * I + 1) * nz;
      int64_t c01 = ((int64_t)(2 * J + 1) * f->nx + 2 * I) * nz;
      int64_t c11 = ((int64_t)(2 * J + 1) * f->nx + 2 * I + 1) * nz;
      int64_t cc = ((int64_t)J * nxc + I) * nz;
      for (int k = 0; k < nz; ++k) rc[cc + k] = rf[c00 + k] + rf[c10 + k] + rf[c01 + k] + rf[c11 + k];
    }
}

/* x_f += P e_c: every fine column gets the value of its coarse column. */
static void mg_prolong_add(const grid_t* f, const double* ec, double* xf) {
  int nxc = f->nx / 2, nz = f->nz;
  for (int j = 0; j < f->ny; ++j)
    for (int i = 0; i < f->nx; ++i) {
      int64_t cf = ((int64_t)j * f->nx + i) * nz;
      int64_t cc = ((int64_t)(j / 2) * nxc + i / 2) * nz;
      for (int k = 0; k < nz; ++k) xf[cf + k] += ec[cc + k];
    }
}

/* One damped line-relaxation step on level l: x += omega M^{-1} (b - A x). */
static int mg_smooth(mg_t* mg, int l) {
  const grid_t* g = &mg->g[l];
  int64_t n = (int64_t)g->nx * g->ny * g->nz;
  double *b = mg->b[l], *x = mg->x[l], *t = mg->t[l], *z = mg->z[l];
  apply_A(g, x, t);
  for (int64_t i = 0; i < n; ++i) t[i] = b[i] - t[i];
  int st = precond(g, t, z, mg->phi, mg->y);
  if (st) return st;
  for (int64_t i = 0; i < n; ++i) x[i] += mg->omega * z[i];
  return ORACLE_OK;
}

/* x_l = V_l(b_l). */
static int mg_vcycle(mg_t* mg, int l) {
  const grid_t* g = &mg->g[l];
  int64_t n = (int64_t)g->nx * g->ny * g->nz;
  memset(mg->x[l], 0, sizeof(double) * n);
  for (int s = 0; s < mg->nu; ++s) {
    int st = mg_smooth(mg, l);
    if (st) return st;
  }
  if (l == mg->nlev - 1) return ORACLE_OK;
  apply_A(g, mg->x[l], mg->t[l]);
  for (int64_t i = 0; i < n; ++i) mg->t[l][i] = mg->b[l][i] - mg->t[l][i];
  mg_restrict(g, mg->t[l], mg->b[l + 1]);
  int st = mg_vcycle(mg, l + 1);
  if (st) return st;
  mg_prolong_add(g, mg->x[l + 1], mg->x[l]);
  for (int s = 0; s < mg->nu; ++s) {
    st = mg_smooth(mg, l);
    if (st) return st;
  }
  return ORACLE_OK;
}

static void mg_free(mg_t* mg) {
  for (int l = 0; l < mg->nlev; ++l) {
    if (l > 0) free(mg->ah[l]);
    free(mg->b[l]); free(mg->x[l]); free(mg->t[l]); free(mg->z[l]);
  }
  free(mg->phi); free(mg->y);
}

static int mg_init(mg_t* mg, const grid_t* g0, int nu, double omega, int max_levels) {
  memset(mg, 0, sizeof(*mg));
  if (nu < 1 || !(omega > 0.0)) return ORACLE_EINVAL;
  mg->nu = nu;
  mg->omega = omega;
  mg->nlev = mg_count_levels(g0->nx, g0->ny, max_levels);
  mg->phi = (double*)malloc(sizeof(double) * g0->nz);
  mg->y = (double*)malloc(sizeof(double) * g0->nz);
  int bad = !mg->phi || !mg->y;
  for (int l = 0; l < mg->nlev && !bad; ++l) {
    if (l == 0) {
      mg->g[0] = *g0;
    } else {
      const grid_t* f = &mg->g[l - 1];
      mg->ah[l] = (double*)malloc(sizeof(double) * (f->nx / 2) * (f->ny / 2));
      if (!mg->ah[l]) { bad = 1; break; }
      mg_coarse_ah(f->nx, f->ny, f->ah, mg->ah[l]);
      grid_t c = {f->nx / 2, f->ny / 2, f->nz, mg->ah[l], f->a_v, f->mass, f->h, 4.0 * f->area};
      mg->g[l] = c;
    }
    int64_t n = (int64_t)mg->g[l].nx * mg->g[l].ny * mg->g[l].nz;
    mg->b[l] = (double*)malloc(sizeof(double) * n);
    mg->x[l] = (double*)malloc(sizeof(double) * n);
    mg->t[l] = (double*)malloc(sizeof(double) * n);
    mg->z[l] = (double*)malloc(sizeof(double) * n);
    bad = !mg->b[l] || !mg->x[l] || !mg->t[l] || !mg->z[l];
  }
  if (bad) {
    mg_free(mg);
    return ORACLE_ENOMEM;
  }
  return ORACLE_OK;
}

static int mg_prec(void* c, const double* r, double* z) {
  mg_t* mg = (mg_t*)c;
  const grid_t* g = &mg->g[0];
  int64_t n = (int64_t)g->nx * g->ny * g->nz;
  memcpy(mg->b[0], r, sizeof(double) * n);
  int st = mg_vcycle(mg, 0);
  if (st) return st;
  memcpy(z, mg->x[0], sizeof(double) * n);
  return ORACLE_OK;
}

/* Number of multigrid levels of an nx x ny grid (max_levels <= 0: no cap). */
int oracle_mg_levels(int nx, int ny, int max_levels) {
  if (nx < 1 || ny < 1) return 0;
  return mg_count_levels(nx, ny, max_levels);
}

/* a_h of level `level` (nx/2^level x ny/2^level values, index J*nxc+I). */
int oracle_mg_level_ah(int nx, int ny, const double* ah, int level, double* ah_out) {
  if (nx < 1 || ny < 1 || !ah || !ah_out || level < 0 || level >= mg_count_levels(nx, ny, 0))
    return ORACLE_EINVAL;
  int cx = nx, cy = ny;
  double* cur = (double*)malloc(sizeof(double) * (size_t)nx * ny);
  double* nxt = (double*)malloc(sizeof(double) * (size_t)nx * ny);
  if (!cur || !nxt) { free(cur); free(nxt); return ORACLE_ENOMEM; }
  memcpy(cur, ah, sizeof(double) * (size_t)nx * ny);
  for (int l = 0; l < level; ++l) {
    mg_coarse_ah(cx, cy, cur, nxt);
    cx /= 2;
    cy /= 2;
    double* tmp = cur; cur = nxt; nxt = tmp;
  }
  memcpy(ah_out, cur, sizeof(double) * (size_t)cx * cy);
  free(cur); free(nxt);
  return ORACLE_OK;
}

/* y = A x on a grid of horizontal cell area `area` (the level operator). */
int oracle_apply_A_area(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                        const double* h, double area, const double* x, double* y) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, area};
  if (check_grid(&g) || !x || !y || !(area > 0.0)) return ORACLE_EINVAL;
  apply_A(&g, x, y);
  return ORACLE_OK;
}

/* The intergrid operators between an nx x ny x nz grid and its coarsening
 * (nx, ny even): rc = R rf, and xf += P ec. */
int oracle_mg_restrict(int nx, int ny, int nz, const double* rf, double* rc) {
  grid_t g = {nx, ny, nz, rf, 0.0, 0.0, rf, 1.0};
  if (nx < 2 || ny < 2 || nx % 2 || ny % 2 || nz < 1 || !rf || !rc) return ORACLE_EINVAL;
  mg_restrict(&g, rf, rc);
  return ORACLE_OK;
}

int oracle_mg_prolong_add(int nx, int ny, int nz, const double* ec, double* xf) {
  grid_t g = {nx, ny, nz, ec, 0.0, 0.0, ec, 1.0};
  if (nx < 2 || ny < 2 || nx % 2 || ny % 2 || nz < 1 || !ec || !xf) return ORACLE_EINVAL;
  mg_prolong_add(&g, ec, xf);
  return ORACLE_OK;
}

/* z = B r, one V-cycle. */
int oracle_mg_vcycle(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                     const double* h, int nu, double omega, int max_levels, const double* r,
                     double* z) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
  if (check_grid(&g) || !r || !z) return ORACLE_EINVAL;
  mg_t mg;
  int st = mg_init(&mg, &g, nu, omega, max_levels);
  if (st) return st;
  st = mg_prec(&mg, r, z);
  mg_free(&mg);
  return st;
}

/* PCG preconditioned by one V-cycle per iteration. */
int oracle_mg_pcg(int nx, int ny, int nz, const double* ah, double a_v, double mass,
                  const double* h, int nu, double omega, int max_levels, const double* b,
                  double* x, double rtol, int maxit, int* iters, double* hist) {
  grid_t g = {nx, ny, nz, ah, a_v, mass, h, 1.0};
  if (check_grid(&g) || !b || !x || !iters || maxit < 0 || !(rtol >= 0.0)) return ORACLE_EINVAL;
  mg_t mg;
  int st = mg_init(&mg, &g, nu, omega, max_levels);
  if (st) return st;
  st = pcg_loop(&g, mg_prec, &mg, b, x, rtol, maxit, iters, hist);
  mg_free(&mg);
  return st;
}
