/*
 * pcg.h -- C ABI of libpcg: a matrix-free preconditioned conjugate gradient
 * (PCG) solver, in fp64 on one GB300 GPU (sm_103a), for strongly vertically
 * anisotropic 3D elliptic operators on flat tensor-product grids.
 *
 * The method is that of E. Mueller, X. Guo, R. Scheichl, S. Shi, "Matrix-free
 * GPU implementation of a preconditioned conjugate gradient solver for
 * anisotropic elliptic PDEs" (2013):
 *   - the operator is applied matrix-free, the 7-point stencil recomputed from
 *     a few per-level and per-column coefficients (section 4.2, eq. (18));
 *   - the preconditioner solves one tridiagonal system exactly per vertical
 *     column with the Thomas algorithm (section 4.1, eq. (19));
 *   - the PCG iteration is loop-fused into two sweeps over the grid per
 *     iteration, each carrying its own inner products (section 4.3,
 *     Algorithm 1; Appendix A, Algorithms 2 and 3).
 *
 * Operator.  On an nx x ny x nz grid, periodic in the horizontal (i, j),
 * homogeneous Neumann at the bottom (k = 0) and top (k = nz-1), with layer
 * thicknesses h_k and unit horizontal cell area and spacing:
 *   (A u)_{ijk} = mass*h_k*u_{ijk}
 *               + h_k * sum_{4 faces f} a_f (u_{ijk} - u_{nbr(f),k})
 *               + T_{k+1/2} (u_{ijk} - u_{ij,k+1})   [k < nz-1]
 *               + T_{k-1/2} (u_{ijk} - u_{ij,k-1})   [k > 0]
 * with T_{k+1/2} = a_v / (0.5*(h_k + h_{k+1})) and a_f the mean of a_h over
 * the two cells of face f (section 3, eqs. (5)-(8)).  A is symmetric
 * positive definite when mass > 0.  The preconditioner M keeps, per column,
 * the vertical couplings and the full diagonal and drops every coupling to
 * the horizontal neighbours (eq. (19)).
 *
 * Layout.  Every vector is nx*ny*nz fp64 values, vertical index fastest:
 * cell (i, j, k) is at ((j*nx) + i)*nz + k (section 3, eq. (10)).
 *
 * Devices and streams.  A context lives on the CUDA device that is current
 * when pcg_create is called; every later call must be made with that device
 * current.  Device pointers must point to memory of that device.  All work
 * is enqueued on the context's stream (pcg_set_stream; default: the legacy
 * default stream).
 *
 * Errors.  Every function returns a status code (pcg_status) and never
 * aborts, exits or prints.  On failure, pcg_last_error() gives a message.
 * Argument errors are detected on the host before any work is enqueued,
 * except the values of an a_h field passed to pcg_update_coeffs or
 * pcg_update_solve_host(_async): those are copied to a staging buffer and
 * checked there on the device; a rejected field leaves the context as it
 * was.
 */
#ifndef PCG_H
#define PCG_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PCG_OK = 0,          /* success */
  PCG_EINVAL = 1,      /* invalid argument (sizes, NULL pointers, coefficients, rtol, maxit) */
  PCG_ENOMEM = 2,      /* device or pinned-host allocation failed */
  PCG_ECUDA = 3,       /* a CUDA runtime call failed (no device, launch error, ...) */
  PCG_ENOTCONV = 4,    /* rtol > 0 and maxit iterations did not reach it */
  PCG_EBREAKDOWN = 5,  /* <p,Ap> <= 0, <r,z> <= 0 or a non-finite residual (NaN/Inf input) */
  PCG_ETIMEOUT = 6     /* a bounded device wait (a grid barrier of the persistent loop) ran out; reported by pcg_solve */
} pcg_status;

typedef struct pcg_ctx pcg_ctx; /* opaque; owns every internal device buffer */

/* Coefficients of the operator.  All host pointers are read during the call
 * (pcg_create / pcg_update_coeffs) and copied; the caller keeps ownership. */
typedef struct {
  double a_h;              /* constant horizontal coefficient (>= 0), used when a_h_field == NULL */
  const double* a_h_field; /* host, nx*ny values a_h(i,j) >= 0 at index j*nx+i, or NULL */
  double a_v;              /* vertical coefficient (>= 0) */
  double mass;             /* zero-order coefficient (> 0) */
  const double* dz;        /* host, nz layer thicknesses h_k > 0 (k = 0 is the bottom), or NULL for all 1 */
} pcg_coeffs;

/* Create a solver context for an nx x ny x nz grid on the current device.
 * Copies the coefficients, builds the per-level tables on the host and the
 * per-column / per-cell tables (face coefficients, diagonal, Thomas factors)
 * on the device (section 4.2: "four vectors ... copied to the device once"),
 * and allocates the workspace r, z, p, q.  Synchronous.
 * Sizes: nx, ny, nz >= 1, nx*ny*nz < 2^40.  *out receives the context, or
 * NULL on failure.  Errors: PCG_EINVAL, PCG_ENOMEM, PCG_ECUDA. */
int pcg_create(int nx, int ny, int nz, const pcg_coeffs* coeffs, pcg_ctx** out);

/* Free every resource of the context.  NULL-safe.  Synchronises its stream. */
void pcg_destroy(pcg_ctx* ctx);

/* Replace the coefficients of an existing context without any allocation
 * (same grid).  A context created with a constant a_h cannot switch to a
 * field (PCG_EINVAL); the reverse is allowed.  Enqueued on the context's
 * stream: with a constant a_h the call returns without waiting for the
 * device; with an a_h field it returns after the set-up kernels, whose
 * checks it reports (PCG_EINVAL for a bad field value, PCG_EBREAKDOWN for a
 * non-positive Thomas pivot). */
int pcg_update_coeffs(pcg_ctx* ctx, const pcg_coeffs* coeffs);

/* Use `stream` (a cudaStream_t, or NULL for the legacy default stream) for
 * all later work of this context.  Work already queued on the previous
 * stream comes first: the new stream waits for it on the device. */
int pcg_set_stream(pcg_ctx* ctx, void* stream);

/* Layout of the solver's internal vectors (r, z, p, q and a copy of the
 * iterate) during pcg_solve.  The caller's vectors always keep the
 * column-contiguous layout of this header.
 *   PCG_LAYOUT_TILED   (default) horizontal index fastest within tiles of
 *                      32 consecutive columns: cell (column c, level k) at
 *                      (c/32*nz + k)*32 + c%32, the GPU layout of the paper
 *                      (section 6.1, eq. (22)) in blocked form.  b and x are
 *                      converted at the start and the end of each solve; the
 *                      context holds two more vectors for it (one if a_h is
 *                      constant).
 *   PCG_LAYOUT_COLUMN  vertical index fastest, like the caller's vectors
 *                      (section 3 eq. (10)); no conversions.
 * Synchronous.  Errors: PCG_EINVAL (unknown layout), PCG_ENOMEM, PCG_ECUDA. */
enum { PCG_LAYOUT_COLUMN = 0, PCG_LAYOUT_TILED = 1 };
int pcg_set_layout(pcg_ctx* ctx, int layout);

/* Where the sweeps of pcg_solve take the per-cell diagonal and the Thomas
 * factors T_{k+1/2}/D_k and 1/D_k of an a_h field (eqs. (18)-(19)) from:
 *   PCG_FACTORS_STORED     (default) the per-cell arrays that pcg_create and
 *                          pcg_update_coeffs compute once: 24 bytes per cell
 *                          read in every iteration;
 *   PCG_FACTORS_RECOMPUTE  rebuilt in every sweep from the per-level table and
 *                          the face values, as the paper's Algorithm 3 does:
 *                          no per-cell reads, but a division, a reciprocal and
 *                          about six more fp64 operations per cell.
 * Both give bit for bit the same iterates (the rebuilt numbers are rounded
 * like the set-up rounds them).  RECOMPUTE applies to the row-tiled layout
 * with an a_h field; in the column layout, or with a constant a_h (whose
 * factors are per level), the stored path runs.  The first switch to
 * RECOMPUTE allocates a scratch of 32*nz doubles per resident warp of the
 * preconditioner sweep.  Synchronous with the host only through that
 * allocation.  Errors: PCG_EINVAL (unknown mode), PCG_ENOMEM, PCG_ECUDA. */
enum { PCG_FACTORS_STORED = 0, PCG_FACTORS_RECOMPUTE = 1 };
int pcg_set_factors(pcg_ctx* ctx, int mode);

/* How the preconditioner sweep of the row-tiled layout solves each column
 * system of M (eq. (19)):
 *   nblocks = 1        one thread walks the whole column (Thomas algorithm);
 *   nblocks = 2,4,8,16 substructuring (section 6.1): the column is cut into
 *                      nblocks blocks by nblocks-1 interface levels; the
 *                      blocks are solved independently by different warps,
 *                      then the interface (Schur complement) system, then
 *                      the blocks are corrected.  Same M^{-1} r up to
 *                      rounding (a few units of cond(T) * eps); more
 *                      parallelism for grids with few columns.  Needs
 *                      nz >= 2*nblocks-1 and 256*(2*nz+4*nblocks+1) bytes
 *                      of shared memory per block of nblocks warps;
 *   nblocks = 0        (default) automatic: 4 (or 2) blocks only for grids
 *                      with fewer tiles of 32 columns than half the SMs,
 *                      where the sweep is latency-bound, and only when the
 *                      persistent loop (pcg_set_loop) does not take them,
 *                      which is faster still there; else 1.  (The
 *                      substructured sweep does 8 fp64 operations per cell
 *                      against 6, and the fp64 rate bounds larger grids.)
 * The substructured sweep keeps its own per-cell tables (four doubles per
 * cell, rebuilt by pcg_update_coeffs); it takes precedence over
 * PCG_FACTORS_RECOMPUTE.  The column layout always uses Thomas.  Synchronous.
 * Errors: PCG_EINVAL (bad nblocks, columns too tall), PCG_ENOMEM, PCG_ECUDA,
 * PCG_EBREAKDOWN (a pivot of the block or interface system is not
 * positive). */
int pcg_set_substructuring(pcg_ctx* ctx, int nblocks);

/* How pcg_solve drives the iterations in the row-tiled layout:
 *   PCG_LOOP_BATCHED     the two fused sweeps of every iteration are kernel
 *                        launches, enqueued in batches (one CUDA graph each);
 *                        the host polls the device's completion flag one batch
 *                        behind;
 *   PCG_LOOP_PERSISTENT  one cooperative kernel runs all iterations: the same
 *                        two sweeps, separated by grid-wide barriers, every
 *                        block taking the scalar decisions from the same
 *                        fixed-order sums; for grids too small to fill the
 *                        GPU, where launch latency dominates an iteration.  A
 *                        barrier wait that runs out (about a second) ends the
 *                        solve with PCG_ETIMEOUT;
 *   PCG_LOOP_CLUSTER     one thread-block cluster (16 CTAs, or 8) runs all
 *                        iterations with every vector of the solve in its
 *                        distributed shared memory: the stencil sweep reads
 *                        the neighbouring tiles' z from the owning CTA's shared
 *                        memory, partial sums go to every CTA's shared memory,
 *                        and hardware cluster barriers separate the sweeps; for
 *                        grids that fit (about 40 K cells with an a_h field,
 *                        70 K with a constant one);
 *   PCG_LOOP_AUTO        (default) the cluster loop where the grid fits,
 *                        else persistent for grids with fewer tiles of 32
 *                        columns than 4 per SM, or than 16 per SM with at
 *                        most 6 * 2^20 cells, else batched.
 * The persistent and cluster loops need Thomas column solves (no
 * substructuring), stored factors and the line preconditioner; the cluster
 * loop also the residual form of A z (pcg_set_az_form), and a device that
 * launches clusters.  The persistent loop needs cooperative launches.  Where a
 * loop cannot run, the next one in the order above does.  The column layout
 * always runs batched.  Errors: PCG_EINVAL (unknown mode). */
enum { PCG_LOOP_AUTO = 0, PCG_LOOP_BATCHED = 1, PCG_LOOP_PERSISTENT = 2, PCG_LOOP_CLUSTER = 3 };
int pcg_set_loop(pcg_ctx* ctx, int mode);

/* The loop the next pcg_solve will run: PCG_LOOP_BATCHED,
 * PCG_LOOP_PERSISTENT or PCG_LOOP_CLUSTER.  Errors: PCG_EINVAL (NULL). */
int pcg_get_loop(const pcg_ctx* ctx, int* mode_out);

/* How the stencil sweep of pcg_solve forms A z (Appendix A, Algorithm 2:
 * q = A z + beta q):
 *   PCG_AZ_STENCIL   the full 7-point stencil of eq. (18), as the paper's
 *                    sweep computes it: 7 fp64 operations per cell for A z;
 *   PCG_AZ_RESIDUAL  A z = r + (A - M) z.  The preconditioner sweep of the
 *                    same iteration has just solved M z = r (eq. (19)), and
 *                    M holds the whole diagonal of A and its vertical
 *                    couplings, so A z - r is the sum over the four
 *                    horizontal neighbours alone: 4 fp64 operations per
 *                    cell, r read in place of the diagonal.  Equal in exact
 *                    arithmetic; in floating point q differs by the column
 *                    solve's backward error, of the same order (eps |A||z|)
 *                    as the stencil's own rounding;
 *   PCG_AZ_AUTO      (default) RESIDUAL wherever it applies.
 * RESIDUAL needs Thomas column solves (no substructuring, and the line
 * preconditioner); elsewhere the full stencil runs.  Both layouts have both
 * forms.  pcg_apply_A always evaluates the full stencil.  Errors: PCG_EINVAL
 * (unknown form). */
enum { PCG_AZ_AUTO = 0, PCG_AZ_STENCIL = 1, PCG_AZ_RESIDUAL = 2 };
int pcg_set_az_form(pcg_ctx* ctx, int form);

/* The form of A z the next pcg_solve will use: PCG_AZ_STENCIL or
 * PCG_AZ_RESIDUAL.  Errors: PCG_EINVAL (NULL). */
int pcg_get_az_form(const pcg_ctx* ctx, int* form_out);

/* Preconditioner of pcg_solve:
 *   PCG_PREC_LINE       (default) the column (vertical line) solve M^{-1} of
 *                       eq. (19), one Thomas solve per column;
 *   PCG_PREC_MULTIGRID  one V-cycle of tensor-product multigrid per
 *                       iteration, with the column solve as its smoother
 *                       (sections 1, 2 and 9 of the paper name the method
 *                       and leave its intergrid operators open).  Level l+1
 *                       merges the 2x2 columns of level l and keeps all nz
 *                       layers; level l is eqs. (5)-(8) on cells of
 *                       horizontal area 4^l, with a_h averaged over the
 *                       merged columns; prolongation copies a coarse column
 *                       into its 4 fine columns and restriction sums them;
 *                       the smoother is x <- x + omega M_l^{-1} (b - A_l x);
 *                       the cycle smooths nu times from x = 0, corrects from
 *                       the next level, and smooths nu times (the coarsest
 *                       level only smooths).  The cycle is symmetric, so CG
 *                       stays valid; it needs far fewer iterations (11 against
 *                       37 on the graded 1024x1024x128 workload) at about
 *                       three times the work per iteration.
 * Multigrid needs the row-tiled layout (PCG_EINVAL otherwise; switching the
 * layout away is refused while it is selected) and a grid with even nx and
 * ny.  It allocates its levels (about 1/3 of the grid's vectors and tables,
 * plus two fine vectors) and uses stored factors, Thomas smoothing and the
 * batched loop whatever pcg_set_factors, pcg_set_substructuring and
 * pcg_set_loop ask for; its stencil sweep evaluates the full stencil.
 * pcg_update_coeffs rebuilds its levels.  Synchronous.  Errors: PCG_EINVAL,
 * PCG_ENOMEM, PCG_ECUDA, PCG_EBREAKDOWN (a pivot on some level). */
enum { PCG_PREC_LINE = 0, PCG_PREC_MULTIGRID = 1 };
int pcg_set_preconditioner(pcg_ctx* ctx, int prec);

/* Multigrid parameters: nu smoothing steps before and after the coarse
 * correction (1..16, default 1), damping omega in (0, 1] (default 0.8), at
 * most max_levels levels (0, the default: coarsen while nx and ny are even).
 * With multigrid selected, a new max_levels rebuilds the levels.
 * Errors: PCG_EINVAL, PCG_ENOMEM, PCG_ECUDA. */
int pcg_set_multigrid(pcg_ctx* ctx, int nu, double omega, int max_levels);

/* Levels of the multigrid preconditioner in use (0 when it is not
 * selected).  Errors: PCG_EINVAL (NULL). */
int pcg_get_multigrid(const pcg_ctx* ctx, int* levels_out);

/* z = B r, one V-cycle of the multigrid preconditioner, standalone (it must
 * be selected).  r_dev, z_dev: device, N values each in the caller's layout,
 * must not overlap.  Asynchronous.  Errors: PCG_EINVAL, PCG_ECUDA. */
int pcg_mg_vcycle(pcg_ctx* ctx, const double* r_dev, double* z_dev);

/* Test hook for the persistent loop's bounded waits: with absent > 0, its
 * grid barriers count `absent` arrivals that never come, so the first
 * barrier wait of the next persistent solve runs out (about a second) and the
 * solve returns PCG_ETIMEOUT; the context stays usable.  0 (default) is
 * normal operation.  Nothing faults or waits without bound.
 * Errors: PCG_EINVAL (NULL, absent < 0). */
int pcg_test_barrier_absent(pcg_ctx* ctx, int absent);

/* Test hook: fills the solver's own work vectors (r, z, p, q and the row-tiled
 * iterate, padding included) with NaN, as memory that an earlier user left
 * behind may hold.  A solve writes each of them before it reads it, so its
 * results do not depend on what they held.  Asynchronous, on the context's
 * stream; the caller's vectors are not touched.
 * Errors: PCG_EINVAL (NULL), PCG_ECUDA. */
int pcg_test_poison_work(pcg_ctx* ctx);

/* Test hook for the column solves on column-contiguous vectors (pcg_precond
 * and the column layout's preconditioner sweep): enable = 0 makes them take
 * the kernels that keep the forward pass's w in global memory instead of in
 * the SM's tensor memory, so that both can be checked and timed; 1 (default)
 * takes the tensor-memory kernels wherever they apply (nz = 32, 64, 128,
 * 16-byte aligned vectors) and the device allows them.
 * Errors: PCG_EINVAL (NULL). */
int pcg_test_tensor_memory(pcg_ctx* ctx, int enable);

/* Blocks per column the row-tiled preconditioner sweep currently uses
 * (1: Thomas), after the automatic choice.  Errors: PCG_EINVAL (NULL). */
int pcg_get_substructuring(const pcg_ctx* ctx, int* nblocks_out);

/* y = A x, the matrix-free 7-point stencil of eq. (18), standalone.
 * x_dev, y_dev: device, N values each, must not overlap.  Asynchronous. */
int pcg_apply_A(pcg_ctx* ctx, const double* x_dev, double* y_dev);

/* z = M^{-1} r, one Thomas solve per column (eq. (19)), standalone.
 * r_dev, z_dev: device, N values each, must not overlap.  Asynchronous. */
int pcg_precond(pcg_ctx* ctx, const double* r_dev, double* z_dev);

/* Solve A x = b by interleaved PCG (Algorithm 1 with the fused sweeps of
 * Algorithms 2 and 3).
 *   b_dev       device, N values (read only).
 *   x_dev       device, N values: the initial guess on entry, the solution
 *               on return (also on PCG_ENOTCONV / PCG_EBREAKDOWN: the last
 *               iterate).  Must not overlap b_dev.
 *   rtol        stop at the first k with ||r_k|| / ||r_0|| < rtol (2-norm of
 *               the recursively updated residual); rtol = 0 runs exactly
 *               maxit iterations.  An exactly zero residual also stops.
 *   maxit       >= 0, at most this many products A p.
 *   iters_out   (may be NULL) number of products A p performed.
 *   res_hist    (host, may be NULL) maxit+1 values; entries 0..iters receive
 *               ||r_k|| / ||r_0|| (0 when r_0 = 0).
 * The whole iteration runs on the context's stream; the host only polls a
 * completion flag between batches.  Returns after the result is in x_dev
 * and res_hist (synchronous on the stream).
 * Errors: PCG_EINVAL, PCG_ECUDA, PCG_ENOTCONV, PCG_EBREAKDOWN. */
int pcg_solve(pcg_ctx* ctx, const double* b_dev, double* x_dev, double rtol, int maxit,
              int* iters_out, double* res_hist);

/* As pcg_solve from the initial guess x0 = 0: x_dev receives the solution
 * and is never read, so neither the caller nor the library fills or scans it
 * first.  Same arguments, stream semantics and errors as pcg_solve. */
int pcg_solve_from_zero(pcg_ctx* ctx, const double* b_dev, double* x_dev, double rtol,
                        int maxit, int* iters_out, double* res_hist);

/* As pcg_solve, with b and x in HOST memory: copies b and x in, solves,
 * copies x out (section 6: the host copies the initial solution and the
 * right-hand side in and the solution out).  The device copies of b and x
 * are allocated on the first call and kept by the context.  Page-locked
 * host memory gives the fastest transfers; pageable memory also works. */
int pcg_solve_host(pcg_ctx* ctx, const double* b_host, double* x_host, double rtol,
                   int maxit, int* iters_out, double* res_hist);

/* As pcg_solve_host, with the initial guess separate from the output:
 *   x0_host  (host, may be NULL) the initial guess; NULL means x0 = 0 (set on
 *            the device: nothing is copied in for it); may equal x_host;
 *   x_host   (host) receives the solution; with x0_host == NULL or another
 *            buffer it is written only.
 * A caller solving repeatedly from x0 = 0 can so keep one page-locked output
 * buffer: no host memset, and one copy in instead of two.
 * Errors: as pcg_solve_host; PCG_EINVAL also when x0 overlaps b. */
int pcg_solve_host_x0(pcg_ctx* ctx, const double* b_host, const double* x0_host, double* x_host,
                      double rtol, int maxit, int* iters_out, double* res_hist);

/* pcg_update_coeffs followed by pcg_solve_host_x0, in one call, for callers
 * that replace the coefficients before every solve: the copies of b and x0
 * go in on a second stream of the context while the set-up kernels of the
 * new coefficients run (section 6: the vertical coefficient vectors and the
 * right-hand side are copied to the device, the solution back).
 *   coeffs   as pcg_update_coeffs (read during the call);
 *   b_host, x0_host, x_host, rtol, maxit, iters_out, res_hist
 *            as pcg_solve_host_x0.
 * b_host and x0_host must hold their values when the call is made: they are
 * read at once, not after earlier work on the context's stream.  With
 * page-locked host memory the host-to-device copies overlap the set-up; with
 * pageable memory the host copies while the set-up runs.  Synchronous.
 * Errors: those of pcg_update_coeffs (checked first; on PCG_EBREAKDOWN for a
 * non-positive pivot nothing is solved) and of pcg_solve_host_x0. */
int pcg_update_solve_host(pcg_ctx* ctx, const pcg_coeffs* coeffs, const double* b_host,
                          const double* x0_host, double* x_host, double rtol, int maxit,
                          int* iters_out, double* res_hist);

/* As pcg_update_solve_host, but the solution's copy to x_host is left
 * running when the call returns, so that it overlaps the next call's
 * set-up and solve (a caller solving a sequence of systems hides the
 * device-to-host copy of each solution behind the next solve).  The
 * iteration count, the history and the status are final on return; x_host
 * is written by a copy on a stream of the context and must be neither read
 * nor freed before pcg_host_wait (or any synchronous host-buffer call on the
 * context, which waits first) returns.  Consecutive calls alternate between
 * two device copies of x, so the copy of one call's solution and the next
 * call's solve do not touch the same memory; the first call allocates the
 * second copy and the stream.  b_host and x0_host may be the x_host of an
 * earlier call whose copy is still running (a sequence in which each solve
 * starts from the last solution): the copy-in then waits for that copy on the
 * device.  Errors: as pcg_update_solve_host; an error of a copy left running
 * is reported by pcg_host_wait. */
int pcg_update_solve_host_async(pcg_ctx* ctx, const pcg_coeffs* coeffs, const double* b_host,
                                const double* x0_host, double* x_host, double rtol, int maxit,
                                int* iters_out, double* res_hist);

/* Waits until the solution copies left running by pcg_update_solve_host_async
 * have reached their host buffers.  Errors: PCG_EINVAL (NULL), PCG_ECUDA (a
 * copy failed). */
int pcg_host_wait(pcg_ctx* ctx);

/* z = M^{-1} r and *rz_dev = <r, z>, without allocating anything.
 * The paper has no counterpart: this entry point exists for callers that
 * must not allocate device memory while they run -- for instance code that
 * must not synchronise the device (cudaFree does, cudaMalloc may), or
 * applications that hand all device memory to their own pool at start-up
 * and leave none for a library to take.  The context
 * (made earlier with pcg_create) supplies the operator tables; the only
 * scratch, one partial sum per tile of 32 columns, comes from a fixed array
 * of 65,536 doubles (512 KB) compiled into the library, which every GPU that
 * loads the library holds until the process exits.
 *   r_dev, z_dev  device, N values each, must not overlap.
 *   rz_dev        device, 1 value: receives <r, z>; must not lie inside r or z.
 * Grids of more than 65,536 x 32 = 2,097,152 columns are rejected with
 * PCG_EINVAL.  pcg_create looks up the device address of the scratch array
 * (cudaGetSymbolAddress, which also loads the array's module on the device),
 * so this call itself neither loads code nor allocates.  All calls share
 * the one array: calls that overlap on the
 * GPU (from two streams or two host threads) race and give wrong results.
 * Asynchronous on the context's stream; calls no cudaMalloc, cudaFree or
 * other allocating routine. */
int pcg_precond_dot_noalloc(pcg_ctx* ctx, const double* r_dev, double* z_dev, double* rz_dev);

/* Message for the last failed call on this context (or of the last failed
 * pcg_create when ctx is NULL).  Never NULL; owned by the library. */
const char* pcg_last_error(const pcg_ctx* ctx);

/* Per-kernel timing.  When enabled, pcg_solve and pcg_update_coeffs record
 * CUDA events around the kernels they launch on the context's stream (the
 * sweeps enqueued after convergence, which return at once, are not counted);
 * pcg_kernel_times then
 * gives, per kernel kind, the summed device time in milliseconds and the
 * number of launches since the last reset (disabled by default; enabling or
 * disabling resets the counters). */
typedef enum {
  PCG_K_PRECOND_FUSED = 0, /* Algorithm 3 sweep: r -= alpha q; z = M^-1 r; <r,r>, <r,z> */
  PCG_K_SPMV_FUSED = 1,    /* Algorithm 2 sweep: u += alpha p; p = z + beta p; q = Az + beta q; <p,q> */
  PCG_K_RESIDUAL = 2,      /* r = b - A x0, p = q = 0, scalar state reset */
  PCG_K_FINALIZE = 3,      /* deferred x += alpha p */
  PCG_K_APPLY_A = 4,       /* standalone stencil */
  PCG_K_PRECOND = 5,       /* standalone Thomas solve */
  PCG_K_SETUP = 6,         /* coefficient set-up kernels of pcg_update_coeffs (face values,
                              per-cell diagonal and Thomas factors), timed together */
  PCG_K_LOOP = 7,          /* persistent solve loop: all iterations of both sweeps */
  PCG_K_PRECOND_FIRST = 8, /* the first Algorithm 3 sweep of a batched row-tiled solve
                              (alpha = 0: r* = r, q not read) */
  PCG_K_SPMV_FIRST = 9,    /* the first Algorithm 2 sweep of a batched row-tiled solve
                              (alpha = beta = 0: p = z, q = Az, u not updated) */
  PCG_K_COUNT = 10
} pcg_kernel_kind;

int pcg_enable_timing(pcg_ctx* ctx, int enable);
int pcg_kernel_times(pcg_ctx* ctx, double* ms_out /* PCG_K_COUNT */,
                     long long* launches_out /* PCG_K_COUNT */);

/* Geometry of the launches (for the roofline accounting of a caller):
 * grid sizes of the fused kernels and the number of kernels pcg_solve
 * launched in its last call. */
int pcg_launch_info(const pcg_ctx* ctx, int* grid_precond, int* grid_spmv,
                    long long* last_solve_launches);

/* Measured fp64 rate of the current device's non-tensor pipe, the bound of
 * the fused sweeps (their work is fp64 fused multiply-adds, products and sums;
 * the paper reports measured rates per kernel, section 7 Table 7).  Runs one
 * warm-up and `launches` timed launches (1..100, about 20 ms each) of a
 * kernel whose threads each carry 8 independent chains of fp64 fused
 * multiply-adds, warps_per_sm warps per SM (1, 2, 3: one block per SM whose
 * warps sit on that many of the SM's four sub-partitions; or a multiple of 4
 * in [4, 64]: blocks of 4 warps), and reports the fastest launch:
 *   *lane_ops_per_s    fp64 lane operations per second (an FMA counts one),
 *   *sm_mhz            median SM clock inside that launch (clock64 against the
 *                      global timer, per block),
 *   *lanes_per_sm_clk  lane operations per SM per clock.
 * Allocates and frees its own small buffers and stream; synchronous.  The
 * error message of a failure is pcg_last_error(NULL).
 * Errors: PCG_EINVAL, PCG_ENOMEM, PCG_ECUDA. */
int pcg_measure_fp64_rate(int warps_per_sm, int launches, double* lane_ops_per_s,
                          double* sm_mhz, double* lanes_per_sm_clk);

#ifdef __cplusplus
}
#endif

#endif /* PCG_H */
