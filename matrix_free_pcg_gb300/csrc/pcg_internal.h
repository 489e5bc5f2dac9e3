// Internal declarations shared by the host driver (pcg_api.cu) and the
// kernel files (pcg_setup.cu, pcg_kernels.cu, pcg_tiled.cu, pcg_split.cu,
// pcg_noalloc.cu).  Not part of the public ABI (include/pcg.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pcg {

// Columns per preconditioner tile: one warp, one thread per vertical column.
constexpr int kTile = 32;
// Threads per block of the stencil sweeps.
constexpr int kSpmvThreads = 256;
// Largest column height whose staged tiles (32 columns) fit in the 227 KB of
// shared memory of one block; taller columns use the unstaged sweep.
constexpr int kMaxStagedNz = 448;

// Per-level coefficient table, kLevCount rows of nz doubles (row-major).
enum LevRow {
  LV_DIAG = 0,  // constant a_h: full diagonal; field: h_k*mass + T_{k+1/2} + T_{k-1/2}
  LV_UP,        // -T_{k+1/2}  (0 at the top)
  LV_DN,        // -T_{k-1/2}  (0 at the bottom)
  LV_HW,        // constant a_h: -h_k*a_h ; field: -h_k
  LV_NPHI,      // constant a_h: T_{k+1/2} / D_k  (minus the Thomas factor phi_k)
  LV_INVD,      // constant a_h: 1 / D_k
  LV_H,         // h_k
  LV_TUP,       // T_{k+1/2}
  LV_TDN,       // T_{k-1/2}
  kLevCount
};

// Operator description handed to every kernel by value.
struct Op {
  int nx, ny, nz;
  int pz;              // nz rounded up to a multiple of 16 (swizzled tile column stride)
  int pt;              // column stride of the bulk-copied tile: >= nz, even, 2 mod 4
  int stream_smem;     // dynamic shared memory of the streaming preconditioner launch
  int fixed;           // 1: nz is 32, 64 or 128 and the height-specialised sweep is used
  int fixed_smem;      // dynamic shared memory of the height-specialised sweep
  double* wscratch;    // height-specialised sweep: 32*nz doubles per block (grid_precond blocks)
  const double* cdiag_t; // field, row-tiled solver layout: diagonal per cell, row-tiled
  const double* cwE_t;   // field, row-tiled: -h_k * (east face value) per cell
  const double* cwN_t;   // field, row-tiled: -h_k * (north face value) per cell
  int recompute;       // field, row-tiled layout: rebuild the diagonal and the Thomas
                       // factors in every sweep instead of reading them per cell
  double* nscratch;    // recompute: T_{k+1/2}/D_k of the tiles in flight, 32*nz doubles
                       // per warp of the preconditioner grid
  int az_resid;        // row-tiled stencil sweep: A z = r + (A - M) z (M z = r from the
                       // preconditioner sweep) instead of the full 7-point stencil
  int tmem;            // the tensor-memory column-solve kernels (pcg_tmem.cu) can be launched
  // substructured column solve (pcg_split.cu), row-tiled tables
  double* sp_nphi;     // per cell: T_{k+1/2}/D_k of the block's own LDL^T (0 at its top)
  double* sp_invd;     // per cell: 1/D_k of the block's LDL^T
  double* sp_ta;       // per cell: T_{s-1/2} (T_i^{-1} e_first)_k
  double* sp_tb;       // per cell: T_{s+m-1/2} (T_i^{-1} e_last)_k
  double* sp_corners;  // per column and block: corners of T_i^{-1} (set-up only)
  double* sp_invdS;    // per column and interface: 1/D of the interface system's LDL^T
  double* sp_nphiS;    // per column and interface: its -S_{j,j+1}/D_j
  long long ncols;     // nx*ny
  long long n;         // ncols*nz
  long long ntiles;    // ceil(ncols / kTile)
  int varying;         // 1: a_h given per column
  const double* lev;   // kLevCount*nz
  const double* ah;    // field: a_h per column
  const double* faceE; // field: face value between (i,j) and (i+1,j), per column
  const double* faceN; // field: face value between (i,j) and (i,j+1), per column
  const double* cdiag; // field: diagonal per cell, vertical index fastest
  const double* tnphi; // field: T_{k+1/2}/D_k per cell, tile-interleaved ((t*nz+k)*32+lane)
  const double* tinvd; // field: 1/D_k per cell, tile-interleaved
};

// Scalars of the interleaved iteration, resident on the device.
struct DevState {
  double alpha;      // step length of the current direction (0 before the first sweep)
  double beta;       // direction update factor for the next sweep
  double kappa_old;  // <r,z> of the previous preconditioner sweep (1 initially)
  double R0;         // ||r_0||^2
  double rtol;
  double last_sigma, last_kappa, last_R;  // diagnostics
  int it;            // preconditioner sweeps completed
  int done;          // 1: stop; every later sweep returns at once
  int status;        // pcg_status of the solve
  int iters;         // products A p performed when the solve stopped
  int maxit;
  unsigned int ticket_m;  // last-block tickets of the two grid reductions
  unsigned int ticket_a;
  int x0_nonzero;    // start of a row-tiled solve: some bit of x0 is set (see
                     // launch_x0_nonzero)
  double mg_R;       // multigrid preconditioner: ||r||^2 of the current iteration, from the
                     // fine level's first smoothing sweep, for the stopping test
  int setup_error;   // a non-positive Thomas pivot was met in the setup kernel
  int dev_error;     // a bounded device wait ran out (pcg_status PCG_ETIMEOUT)
  unsigned int bar_count;  // arrivals at the grid barriers of the persistent solve loop
};

// ---- launchers (set-up: pcg_setup.cu; column-layout sweeps, stencil, residual and final
// update: pcg_kernels.cu); all enqueue on `s` and return the launch error

cudaError_t launch_face_coeffs(const Op& op, double* faceE, double* faceN, cudaStream_t s);
// *err = 1 if some f[i], i < n, is negative, infinite or NaN (err untouched
// otherwise: the caller zeroes it first).
cudaError_t launch_check_field(const double* f, long long n, int* err, cudaStream_t s);
// *dst = *src by one thread (dst: mapped host memory, read after the stream
// synchronises, without a copy engine).
cudaError_t launch_flag_to_host(const int* src, int* dst, cudaStream_t s);
// Per-cell diagonal (column-contiguous, and row-tiled when cdiag_t is not
// NULL), horizontal weights (row-tiled, when cwE_t is not NULL) and Thomas
// factors (row-tiled) of an a_h field, after the face values.
cudaError_t launch_column_setup(const Op& op, DevState* st, double* cdiag, double* cdiag_t,
                                double* cwE_t, double* cwN_t, double* tnphi, double* tinvd,
                                cudaStream_t s);

// r = b - A x ; p = q = 0 ; scalar state reset for a new solve.
cudaError_t launch_residual(const Op& op, DevState* st, const double* b, const double* x,
                            double* r, double* p, double* q, double rtol, int maxit, int grid,
                            cudaStream_t s);
// The same for the row-tiled solver layout, in one launch: r_t = b - A x0,
// u_t = x0 and p_t = q_t = 0 at the row-tiled positions (b and x0 in the
// caller's column-contiguous layout).  With x0_checked, st->x0_nonzero (from
// launch_x0_nonzero) tells whether x0 may be skipped entirely.
// zero_pq: also write p = q = 0 (not needed when the first sweeps of the
// solve are the first-iteration variants, which read neither)
cudaError_t launch_residual_tiled(const Op& op, DevState* st, const double* b, const double* x,
                                  double* r_t, double* u_t, double* p_t, double* q_t, double rtol,
                                  int maxit, bool x0_checked, cudaStream_t s,
                                  bool zero_pq = true);
// st->x0_nonzero = whether any of the n values of x has a bit set (all +0.0:
// the zero initial guess).  Clears the flag first.
cudaError_t launch_x0_nonzero(const double* x, long long n, DevState* st, int num_sms,
                              cudaStream_t s);
// y = A x
cudaError_t launch_apply(const Op& op, const double* x, double* y, int grid, cudaStream_t s);
// z = M^{-1} r  (st receives dev_error if a bounded wait runs out)
cudaError_t launch_precond(const Op& op, DevState* st, const double* r, double* z, int grid,
                           cudaStream_t s);
// Algorithm 3 sweep
cudaError_t launch_precond_fused(const Op& op, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s);
// Algorithm 2 sweep (with op.az_resid: A z from r, the residual M z = r was
// solved for)
cudaError_t launch_spmv_fused(const Op& op, DevState* st, const double* z, const double* r,
                              double* u, double* p, double* q, double* partials, int grid,
                              cudaStream_t s);
// x += alpha p (the update deferred past the last sweep)
cudaError_t launch_finalize(const Op& op, const DevState* st, double* x, const double* p,
                            int grid, cudaStream_t s);

// z = M^{-1} r and *rz = <r, z> with scratch from a fixed device array in
// pcg_noalloc.cu (no allocation); at most kNoallocMaxTiles tiles of 32 columns.
// partials: the array's device address on the current device, from
// noalloc_scratch_address (called with that device current).
constexpr long long kNoallocMaxTiles = 65536;
cudaError_t noalloc_scratch_address(double** out);
cudaError_t launch_precond_dot_noalloc(const Op& op, const double* r, double* z, double* rz,
                                       double* partials, int num_sms, cudaStream_t s);

// Row-tiled solver layout (pcg_tiled.cu): cell (c,k) at (c/32*nz + k)*32 + c%32.
// Row-tiled vectors hold ntiles*32*nz values (the last tile padded to 32
// columns).  dst_t = src_k (the standalone V-cycle's input).
cudaError_t launch_to_tiled(const Op& op, const double* src_k, double* dst_t, cudaStream_t s);
// dst_k = src_t + alpha p_t (alpha from the device state), or a copy when p_t is NULL.
cudaError_t launch_from_tiled(const Op& op, const DevState* st, const double* src_t,
                              const double* p_t, double* dst_k, cudaStream_t s);
// Algorithm 3 / Algorithm 2 sweeps on row-tiled vectors; with op.recompute the
// per-cell diagonal and Thomas factors are rebuilt on the fly (op.nscratch must
// then hold kTmWarpsPerBlock*32*nz doubles per block of grid_tiled_precond).
// first: the first sweep of a solve (alpha = 0, q never written; stored
// factors only)
cudaError_t launch_precond_tiled(const Op& op, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s, bool first = false);
// With op.az_resid the stencil sweep reads r (the residual that the
// preconditioner sweep's z solves M z = r for) instead of the diagonal.
// first: the first sweep of a solve (alpha = beta = 0, p and q never written,
// u holding x0; stored factors only)
cudaError_t launch_spmv_tiled(const Op& op, DevState* st, const double* z, const double* r,
                              double* u, double* p, double* q, double* partials, int grid,
                              cudaStream_t s, bool first = false);
// Warps per block of the row-tiled preconditioner sweep, and its resident
// warps per SM (each warp keeps the w of its tile and the factors the
// backward pass reads again live in L2; 12 per SM keep this within L2 at
// nz = 128 and leave three warps per sub-partition to hide fp64 latency).
constexpr int kTmWarpsPerBlock = 4;
constexpr int kTmWarpsPerSm = 12;
// Whole solve loop of the row-tiled layout (Thomas column solves, stored
// factors) in one cooperative launch: grid_persistent gives its grid (0: not
// available), launch_persistent runs iterations until the stopping test.
int grid_persistent(const Op& op, int num_sms);
cudaError_t launch_persistent(const Op& op, DevState* st, double* r, double* q, double* z,
                              double* u, double* p, double* partials, double* hist, int grid,
                              unsigned int absent, cudaStream_t s);

// Whole solve loop in the shared memory of one thread-block cluster
// (pcg_cluster.cu; row-tiled layout, Thomas column solves, stored factors, A z
// in the residual form): cluster_ctas gives the cluster's CTAs (16 or 8; 0:
// the grid does not fit or clusters are not available), launch_cluster_loop
// runs iterations until the stopping test and leaves u and p row-tiled.
int cluster_ctas(const Op& op);
cudaError_t launch_cluster_loop(const Op& op, DevState* st, double* r, double* u, double* p,
                                double* hist, int ctas, cudaStream_t s);

// Grid sizes (blocks) of the two row-tiled sweeps.
int grid_tiled_precond(const Op& op, int num_sms);
int grid_tiled_spmv(const Op& op, int num_sms);

// Substructured column solve (pcg_split.cu): P blocks per column, P in
// {2, 4, 8, 16}, nz >= 2P-1.  Tables in op.sp_*; set-up after every
// coefficient change; sweep = Algorithm 3 with a block of P warps per tile.
bool split_valid(int nz, int P);
size_t split_smem_bytes(int nz, int P);
int split_grid(const Op& op, int P, int num_sms);  // 0: not launchable
cudaError_t launch_split_setup(const Op& op, int P, DevState* st, cudaStream_t s);
cudaError_t launch_precond_split(const Op& op, int P, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s);

// Tensor-product multigrid preconditioner (pcg_mg.cu), row-tiled vectors on
// every level.  A level is an Op (its own per-level table, and for an a_h
// field its face values and per-cell diagonal, weights and Thomas factors)
// on cells of horizontal area 4^l; coarse level l+1 merges 2x2 columns.
struct MgLevel {
  Op op{};
  double *lev = nullptr, *ah = nullptr, *faceE = nullptr, *faceN = nullptr;
  double *cdiag = nullptr, *cdiag_t = nullptr, *cwE_t = nullptr, *cwN_t = nullptr;
  double *tnphi = nullptr, *tinvd = nullptr;
  double *b = nullptr, *x = nullptr, *y = nullptr;  // right-hand side, two iterates
  int grid_first = 1, grid_smooth = 1;              // blocks of the two Thomas sweeps
};
// x = omega M^{-1} b.  fused (finest level inside the solve): first b <- b -
// alpha q with alpha from the device state and ||b||^2 into st->mg_R; if the
// stopping test passes on it, the scalar step is taken (hist) and the rest of
// the cycle is skipped.
cudaError_t launch_mg_first(const Op& op, DevState* st, double* b, const double* q, double* x,
                            double omega, bool fused, double* partials, double* hist, int grid,
                            cudaStream_t s);
// bc = R (b - A x): per layer, the residuals of the 2x2 fine columns summed.
// first: x = omega M^{-1} b exactly as launch_mg_first left it, so that
// b - A x = (1 - omega) b - (A - M) x.
cudaError_t launch_mg_restrict(const Op& fine, const Op& coarse, const DevState* st,
                               const double* b, const double* x, bool first, double omega,
                               double* bc, int num_sms, cudaStream_t s);
// x += P e: every fine column gets its coarse column's value.
cudaError_t launch_mg_prolong(const Op& fine, const Op& coarse, const DevState* st, double* x,
                              const double* e, int num_sms, cudaStream_t s);
// xout = xin + omega M^{-1} (b - A xin), two launches: the residual into
// xout, then the column solves in place.  fused (finest level, last step):
// <b, xout> reduced and the scalar step of Algorithm 1 taken with st->mg_R.
cudaError_t launch_mg_smooth(const Op& op, DevState* st, const double* b, const double* xin,
                             double* xout, double omega, bool fused, double* partials,
                             double* hist, int grid, int num_sms, cudaStream_t s);
// a_h of a coarse level from the finer one (the mean of the 4 merged columns).
cudaError_t launch_mg_coarse_ah(const Op& fine, const Op& coarse, const double* ahf, double* ahc,
                                int num_sms, cudaStream_t s);
int grid_mg_first(const Op& op, int num_sms);
int grid_mg_smooth(const Op& op, int num_sms);

// Column solves with the forward result in tensor memory (pcg_tmem.cu), for
// the caller's column-contiguous layout: nz in {32, 64, 128} and 16-byte
// aligned vectors (precond_tmem_supported).  One block of 8 warps per SM
// (grid_precond_tmem blocks: at most one per SM and none without a tile,
// never more than grid_precond's), each block holding all of its SM's TMEM
// columns.  fused: the Algorithm 3 sweep (r* = r - alpha q, reductions,
// scalar step); otherwise z = M^{-1} r (q, partials and hist unused).
// prepare_precond_tmem sets the kernels' shared-memory attributes (once per
// device).
bool precond_tmem_supported(const Op& op, const double* r, const double* q, const double* z);
cudaError_t prepare_precond_tmem();
int grid_precond_tmem(const Op& op, int num_sms);
cudaError_t launch_precond_tmem(const Op& op, DevState* st, double* r, const double* q,
                                double* z, double* partials, double* hist, bool fused, int grid,
                                cudaStream_t s);

// fp64 rate probe (pcg_peak.cu): fp64 lane operations one launch of `blocks`
// blocks of `threads` threads and `trips` loop trips performs, and the launch
// (stamps: per block, SM cycles and global-timer nanoseconds).
long long fp64_rate_lane_ops(int blocks, int threads, int trips);
cudaError_t launch_fp64_rate(int blocks, int threads, int trips, double* sink,
                             unsigned long long* stamps, cudaStream_t s);

// Occupancy-derived grid sizes (blocks) for the persistent sweeps.  The
// preconditioner's also fixes op.stream_smem (see pcg_kernels.cu).
int grid_precond(Op& op, int num_sms);
int grid_spmv(const Op& op, int num_sms);
// Shared-memory attribute set-up for the staged preconditioner (once per device).
cudaError_t prepare_kernels(const Op& op);

}  // namespace pcg
