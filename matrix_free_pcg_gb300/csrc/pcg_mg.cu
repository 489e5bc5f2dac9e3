// Tensor-product multigrid preconditioner: the kernels of one V-cycle, on
// row-tiled vectors, cell (column c, level k) at (c/32*nz + k)*32 + c%32 on
// every multigrid level.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// sections 1, 2 and 9: the column solve of eq. (19) as the smoother of a
// geometric multigrid that coarsens only the horizontal directions (the
// tensor-product idea of Boerm and Hiptmair).  The pages leave the intergrid
// operators open; here level l+1 merges the 2x2 columns of level l, the level
// operators are eqs. (5)-(8) on cells of horizontal area 4^l, P copies a
// coarse column into its 4 fine columns, R = P^T sums them, and the smoother
// is the damped line relaxation x <- x + omega M_l^{-1} (b - A_l x).
//
// One V-cycle, per level from the finest down and back up:
//   k_mg_first       x = omega M^{-1} b (on the finest level fused with the
//                    residual update r <- r - alpha q of Algorithm 3 and ||r||^2)
//   smoothing        further steps (nu > 1): k_mg_residual, k_mg_thomas_add
//   k_mg_restrict    b_{l+1} = R (b - A x) (with one smoothing step from zero,
//                    M x = omega b leaves only the horizontal terms of A x)
//   ... the coarser levels ...
//   k_mg_prolong     x += P x_{l+1}
//   smoothing        nu steps (on the finest level the last one also reduces
//                    <r, z> and takes the scalar step of Algorithm 1)
// Every kernel without a recurrence runs one thread per cell, so that the
// small coarse levels are not left to a few threads walking their columns;
// the column solves use the chunked Thomas body of the preconditioner sweep.
#include <algorithm>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"
#include "pcg_sweeps.cuh"

namespace pcg {
namespace {

constexpr int kMgThreads = 256;  // blocks of the one-thread-per-cell kernels

// (A x) at row-tiled offset o (level k, ko = k*32) of a column whose
// neighbours' bases are bE..bS; xd, xc, xu are x at k-1, k, k+1.
template <bool VARY>
__device__ __forceinline__ double stencil_at(const Op& op, const double* __restrict__ x,
                                             long long o, long long ko, int k, long long bE,
                                             long long bW, long long bN, long long bS,
                                             double xd, double xc, double xu) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const double zE = x[bE + ko], zW = x[bW + ko], zN = x[bN + ko], zS = x[bS + ko];
  double a;
  if (VARY) {
    a = op.cdiag_t[o] * xc;
    a = fma(__ldg(lev + LV_UP * nz + k), xu, a);
    a = fma(__ldg(lev + LV_DN * nz + k), xd, a);
    a = fma(op.cwE_t[o], zE, a);
    a = fma(op.cwE_t[bW + ko], zW, a);
    a = fma(op.cwN_t[o], zN, a);
    a = fma(op.cwN_t[bS + ko], zS, a);
  } else {
    const double hs = (zE + zW) + (zN + zS);
    a = __ldg(lev + LV_DIAG * nz + k) * xc;
    a = fma(__ldg(lev + LV_UP * nz + k), xu, a);
    a = fma(__ldg(lev + LV_DN * nz + k), xd, a);
    a = fma(__ldg(lev + LV_HW * nz + k), hs, a);
  }
  return a;
}

// Whether the stopping test of Algorithm 1 ends the solve at this iteration
// from ||r||^2 alone: every outcome of finish_precond_sweep but the <r, z>
// breakdown, evaluated in its order with its expressions.
__device__ __forceinline__ bool stops_on_R(const DevState* st, double R) {
  const int it = st->it;
  const double R0 = (it == 0) ? R : st->R0;
  if (st->dev_error || R0 == 0.0) return true;
  if (!(R < INFINITY) || !(R0 < INFINITY)) return true;
  const double ratio = (R0 > 0.0) ? sqrt(R / R0) : 0.0;
  return ratio < st->rtol || R == 0.0 || it >= st->maxit;
}

// x = omega M^{-1} b, one warp per tile of 32 columns (the Thomas tile body
// of the preconditioner sweep).  FUSED: b <- b - alpha q first, and ||b||^2
// reduced into st->mg_R; when that alone stops the solve, the scalar step is
// taken here, and the rest of the V-cycle returns at once.
template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTmThreads) k_mg_first(Op op, DevState* st,
                                                         double* __restrict__ b,
                                                         const double* __restrict__ q,
                                                         double* __restrict__ x, double omega,
                                                         double* __restrict__ partials,
                                                         double* __restrict__ hist) {
  if (ld_done(st)) return;
  const double nalpha = FUSED ? -st->alpha : 0.0;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accR = 0.0, accK = 0.0;
  for (long long t = warp0; t < op.ntiles; t += nwarps)
    precond_tile<VARY, FUSED, false, true>(op, t, lane, b, q, x, nalpha, keep, stream, accR,
                                           accK, omega);
  if (FUSED) {
    double R, unused;
    if (grid_sum2<kTmThreads>(accR, 0.0, partials, &st->ticket_m, R, unused)) {
      st->mg_R = R;
      if (stops_on_R(st, R)) finish_precond_sweep(st, R, 0.0, hist);
    }
  }
}

// The cell (column c, level k) of row-tiled offset o, or false for a padded
// lane of the last tile.
__device__ __forceinline__ bool tiled_cell(const Op& op, long long o, long long& col, int& k) {
  const long long tk = o >> 5;
  const long long t = tk / op.nz;
  k = (int)(tk - t * op.nz);
  col = t * kTile + (o & (kTile - 1));
  return col < op.ncols;
}

// b - A x at cell (col, k), row-tiled offset o.
template <bool VARY>
__device__ __forceinline__ double residual_at(const Op& op, const double* __restrict__ b,
                                              const double* __restrict__ x, long long col, int k,
                                              long long o) {
  const int nz = op.nz;
  const Nbr nb = neighbours(op, col);
  const long long ko = (long long)k * kTile;
  const double xd = (k > 0) ? x[o - kTile] : 0.0;
  const double xu = (k + 1 < nz) ? x[o + kTile] : 0.0;
  return b[o] - stencil_at<VARY>(op, x, o, ko, k, tiled_base(nb.e, nz), tiled_base(nb.w, nz),
                                 tiled_base(nb.n, nz), tiled_base(nb.s, nz), xd, x[o], xu);
}

// s = b - A x, one thread per cell (no recurrence: every level at once).
template <bool VARY>
__global__ void __launch_bounds__(kMgThreads) k_mg_residual(Op op, const DevState* st,
                                                            const double* __restrict__ b,
                                                            const double* __restrict__ x,
                                                            double* __restrict__ s) {
  if (ld_done(st)) return;
  const long long total = op.ntiles * (long long)op.nz * kTile;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    long long col;
    int k;
    if (tiled_cell(op, o, col, k)) s[o] = residual_at<VARY>(op, b, x, col, k, o);
  }
}

// xout = xin + omega M^{-1} s with s held in xout on entry (one warp per
// tile; the chunked Thomas body of the preconditioner sweep: the operands of
// the next 8 levels are fetched while the current ones compute).  FUSED:
// <b, xout> reduced, then the scalar step of Algorithm 1 with ||r||^2 from
// st->mg_R.
template <bool VARY>
__device__ __forceinline__ void thomas_add_tile(const Op& op, long long t, int lane,
                                                const double* __restrict__ b,
                                                const double* __restrict__ xin,
                                                double* __restrict__ xout, double omega,
                                                uint64_t keep, uint64_t stream, bool fused,
                                                double& accK) {
  const int nz = op.nz;
  const int fs = VARY ? kTile : 1;
  if (t * kTile + lane >= op.ncols) return;
  const long long base = t * nz * kTile + lane;
  double* __restrict__ ot = xout + base;
  const double* __restrict__ xt = xin + base;
  const double* __restrict__ bt = b + base;
  const double* __restrict__ fi = VARY ? op.tinvd + base : op.lev + LV_INVD * nz;
  const double* __restrict__ fn = VARY ? op.tnphi + base : op.lev + LV_NPHI * nz;
  double cs[kTmChunk], ci[kTmChunk], cn[kTmChunk];
#pragma unroll
  for (int j = 0; j < kTmChunk; ++j) {
    const bool in = j < nz;
    cs[j] = in ? ld_hint(ot + j * kTile, stream) : 0.0;
    ci[j] = in ? (VARY ? ld_hint(fi + j * fs, stream) : __ldg(fi + j)) : 0.0;
    cn[j] = in ? (VARY ? ld_hint(fn + j * fs, keep) : __ldg(fn + j)) : 0.0;
  }
  double y = 0.0, nprev = 0.0, w = 0.0;
#pragma unroll 1
  for (int k0 = 0; k0 < nz; k0 += kTmChunk) {
    double ns[kTmChunk], ni[kTmChunk], nn[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = k0 + kTmChunk + j;
      const bool in = k < nz;
      ns[j] = in ? ld_hint(ot + k * kTile, stream) : 0.0;
      ni[j] = in ? (VARY ? ld_hint(fi + k * fs, stream) : __ldg(fi + k)) : 0.0;
      nn[j] = in ? (VARY ? ld_hint(fn + k * fs, keep) : __ldg(fn + k)) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = k0 + j;
      if (k < nz) {
        y = fma(nprev, y, cs[j]);
        w = y * ci[j];
        st_hint(ot + k * kTile, w, keep);
        nprev = cn[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      cs[j] = ns[j];
      ci[j] = ni[j];
      cn[j] = nn[j];
    }
  }
  // back substitution; level k's result is x_k + omega z_k
  double zz = w;
  {
    const long long ko = (long long)(nz - 1) * kTile;
    const double out = fma(omega, zz, xt[ko]);
    st_hint(ot + ko, out, stream);
    if (fused) accK = fma(bt[ko], out, accK);
  }
  double bw[kTmChunk], bn[kTmChunk], bx[kTmChunk], bb[kTmChunk];
#pragma unroll
  for (int j = 0; j < kTmChunk; ++j) {
    const int k = nz - 2 - j;
    bw[j] = (k >= 0) ? ld_hint(ot + k * kTile, stream) : 0.0;
    bn[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
    bx[j] = (k >= 0) ? xt[k * kTile] : 0.0;
    bb[j] = (fused && k >= 0) ? bt[k * kTile] : 0.0;
  }
#pragma unroll 1
  for (int kb = nz - 2; kb >= 0; kb -= kTmChunk) {
    double nw[kTmChunk], nb[kTmChunk], nx[kTmChunk], nbb[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = kb - kTmChunk - j;
      nw[j] = (k >= 0) ? ld_hint(ot + k * kTile, stream) : 0.0;
      nb[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
      nx[j] = (k >= 0) ? xt[k * kTile] : 0.0;
      nbb[j] = (fused && k >= 0) ? bt[k * kTile] : 0.0;
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = kb - j;
      if (k >= 0) {
        zz = fma(bn[j], zz, bw[j]);
        const double out = fma(omega, zz, bx[j]);
        st_hint(ot + k * kTile, out, stream);
        if (fused) accK = fma(bb[j], out, accK);
      }
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      bw[j] = nw[j];
      bn[j] = nb[j];
      bx[j] = nx[j];
      bb[j] = nbb[j];
    }
  }
}

template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTmThreads) k_mg_thomas_add(Op op, DevState* st,
                                                              const double* __restrict__ b,
                                                              const double* __restrict__ xin,
                                                              double* __restrict__ xout,
                                                              double omega,
                                                              double* __restrict__ partials,
                                                              double* __restrict__ hist) {
  if (ld_done(st)) return;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accK = 0.0;
  for (long long t = warp0; t < op.ntiles; t += nwarps)
    thomas_add_tile<VARY>(op, t, lane, b, xin, xout, omega, keep, stream, FUSED, accK);
  if (FUSED) {
    double K, unused;
    if (grid_sum2<kTmThreads>(accK, 0.0, partials, &st->ticket_m, K, unused))
      finish_precond_sweep(st, st->mg_R, K, hist);
  }
}

// b - A x at cell (col, k) for x = omega M^{-1} b (the first smoothing step
// from zero): M x = omega b, and M holds A's diagonal and vertical
// couplings, so b - A x = (1 - omega) b - (A - M) x, the horizontal
// neighbours alone (5 fp64 operations instead of 8).
template <bool VARY>
__device__ __forceinline__ double first_residual_at(const Op& op, const double* __restrict__ b,
                                                    const double* __restrict__ x, double omb,
                                                    long long col, int k, long long o) {
  const int nz = op.nz;
  const Nbr nb = neighbours(op, col);
  const long long ko = (long long)k * kTile;
  const long long bW = tiled_base(nb.w, nz), bS = tiled_base(nb.s, nz);
  const double xE = x[tiled_base(nb.e, nz) + ko], xW = x[bW + ko];
  const double xN = x[tiled_base(nb.n, nz) + ko], xS = x[bS + ko];
  double t = omb * b[o];
  if (VARY) {
    t = fma(-op.cwE_t[o], xE, t);
    t = fma(-op.cwE_t[bW + ko], xW, t);
    t = fma(-op.cwN_t[o], xN, t);
    t = fma(-op.cwN_t[bS + ko], xS, t);
  } else {
    t = fma(-__ldg(op.lev + LV_HW * nz + k), (xE + xW) + (xN + xS), t);
  }
  return t;
}

// bc = R (b - A x): one thread per coarse cell (I, J, k); the residuals of
// the fine columns (2I, 2J), (2I+1, 2J), (2I, 2J+1), (2I+1, 2J+1) at layer k
// summed in that order.  FIRST: x = omega M^{-1} b, the residual from the
// horizontal neighbours alone.
template <bool VARY, bool FIRST>
__global__ void __launch_bounds__(kMgThreads) k_mg_restrict(Op f, Op c, const DevState* st,
                                                            const double* __restrict__ b,
                                                            const double* __restrict__ x,
                                                            double omega,
                                                            double* __restrict__ bc) {
  if (ld_done(st)) return;
  const int nz = f.nz;
  const double omb = 1.0 - omega;
  const long long total = c.ntiles * (long long)nz * kTile;
  for (long long oc = blockIdx.x * (long long)blockDim.x + threadIdx.x; oc < total;
       oc += (long long)gridDim.x * blockDim.x) {
    long long C;
    int k;
    if (!tiled_cell(c, oc, C, k)) continue;
    const long long J = C / c.nx;
    const int I = (int)(C - J * c.nx);
    double t[4];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const long long col = (2 * J + (qd >> 1)) * f.nx + 2 * I + (qd & 1);
      const long long o = tiled_base(col, nz) + (long long)k * kTile;
      t[qd] = FIRST ? first_residual_at<VARY>(f, b, x, omb, col, k, o)
                    : residual_at<VARY>(f, b, x, col, k, o);
    }
    bc[oc] = ((t[0] + t[1]) + t[2]) + t[3];
  }
}

// x += P e: one thread per fine cell (row-tiled order).
__global__ void __launch_bounds__(kMgThreads) k_mg_prolong(Op f, Op c, const DevState* st,
                                                           double* __restrict__ x,
                                                           const double* __restrict__ e) {
  if (ld_done(st)) return;
  const int nz = f.nz;
  const long long total = f.ntiles * (long long)nz * kTile;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(o & (kTile - 1));
    const long long tk = o / kTile;
    const long long t = tk / nz;
    const int k = (int)(tk - t * nz);
    const long long col = t * kTile + lane;
    if (col >= f.ncols) continue;
    const long long j = col / f.nx;
    const int i = (int)(col - j * f.nx);
    const long long C = (j >> 1) * c.nx + (i >> 1);
    x[o] += e[tiled_base(C, nz) + (long long)k * kTile];
  }
}

// a_h of the coarse columns: the mean over the 4 merged fine columns,
// ((a00 + a10) + a01) + a11 times 1/4.
__global__ void __launch_bounds__(kMgThreads) k_mg_coarse_ah(Op f, Op c,
                                                             const double* __restrict__ ahf,
                                                             double* __restrict__ ahc) {
  for (long long C = blockIdx.x * (long long)blockDim.x + threadIdx.x; C < c.ncols;
       C += (long long)gridDim.x * blockDim.x) {
    const long long J = C / c.nx;
    const int I = (int)(C - J * c.nx);
    const long long f0 = 2 * J * f.nx + 2 * I;
    const double sum = ahf[f0] + ahf[f0 + 1] + ahf[f0 + f.nx] + ahf[f0 + f.nx + 1];
    ahc[C] = 0.25 * sum;
  }
}

template <typename K>
int occupancy_grid(K kernel, int threads, int max_per_sm, long long work_blocks, int num_sms) {
  int a = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, kernel, threads, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    a = 1;
  }
  const int per_sm = std::max(1, std::min(a, max_per_sm));
  long long g = std::min<long long>((long long)per_sm * num_sms, work_blocks);
  return (int)std::max<long long>(g, 1);
}

}  // namespace

int grid_mg_first(const Op& op, int num_sms) {
  const long long work = (op.ntiles + kTmWarpsPerBlock - 1) / kTmWarpsPerBlock;
  const int cap = kTmWarpsPerSm / kTmWarpsPerBlock;
  return op.varying ? occupancy_grid(k_mg_first<true, true>, kTmThreads, cap, work, num_sms)
                    : occupancy_grid(k_mg_first<false, true>, kTmThreads, cap, work, num_sms);
}

int grid_mg_smooth(const Op& op, int num_sms) {
  const long long work = (op.ntiles + kTmWarpsPerBlock - 1) / kTmWarpsPerBlock;
  const int cap = kTmWarpsPerSm / kTmWarpsPerBlock;
  return op.varying
             ? occupancy_grid(k_mg_thomas_add<true, true>, kTmThreads, cap, work, num_sms)
             : occupancy_grid(k_mg_thomas_add<false, true>, kTmThreads, cap, work, num_sms);
}

cudaError_t launch_mg_first(const Op& op, DevState* st, double* b, const double* q, double* x,
                            double omega, bool fused, double* partials, double* hist, int grid,
                            cudaStream_t s) {
  if (op.varying) {
    if (fused)
      k_mg_first<true, true><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials, hist);
    else
      k_mg_first<true, false><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials,
                                                             hist);
  } else {
    if (fused)
      k_mg_first<false, true><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials,
                                                             hist);
    else
      k_mg_first<false, false><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials,
                                                              hist);
  }
  return cudaGetLastError();
}

cudaError_t launch_mg_smooth(const Op& op, DevState* st, const double* b, const double* xin,
                             double* xout, double omega, bool fused, double* partials,
                             double* hist, int grid, int num_sms, cudaStream_t s) {
  // the residual into xout, then the column solves in place
  const long long total = op.ntiles * (long long)op.nz * kTile;
  const long long g = std::max<long long>(
      1, std::min<long long>((total + kMgThreads - 1) / kMgThreads, 16LL * num_sms));
  if (op.varying)
    k_mg_residual<true><<<(int)g, kMgThreads, 0, s>>>(op, st, b, xin, xout);
  else
    k_mg_residual<false><<<(int)g, kMgThreads, 0, s>>>(op, st, b, xin, xout);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (op.varying) {
    if (fused)
      k_mg_thomas_add<true, true><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega,
                                                              partials, hist);
    else
      k_mg_thomas_add<true, false><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega,
                                                               partials, hist);
  } else {
    if (fused)
      k_mg_thomas_add<false, true><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega,
                                                               partials, hist);
    else
      k_mg_thomas_add<false, false><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega,
                                                                partials, hist);
  }
  return cudaGetLastError();
}

cudaError_t launch_mg_restrict(const Op& fine, const Op& coarse, const DevState* st,
                               const double* b, const double* x, bool first, double omega,
                               double* bc, int num_sms, cudaStream_t s) {
  const long long total = coarse.ntiles * (long long)coarse.nz * kTile;
  const long long g = std::max<long long>(
      1, std::min<long long>((total + kMgThreads - 1) / kMgThreads, 16LL * num_sms));
  if (first) {
    if (fine.varying)
      k_mg_restrict<true, true><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, omega, bc);
    else
      k_mg_restrict<false, true><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, omega, bc);
  } else {
    if (fine.varying)
      k_mg_restrict<true, false><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, omega, bc);
    else
      k_mg_restrict<false, false><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, omega,
                                                                bc);
  }
  return cudaGetLastError();
}

cudaError_t launch_mg_prolong(const Op& fine, const Op& coarse, const DevState* st, double* x,
                              const double* e, int num_sms, cudaStream_t s) {
  const long long total = fine.ntiles * (long long)fine.nz * kTile;
  const long long g = std::max<long long>(
      1, std::min<long long>((total + kMgThreads - 1) / kMgThreads, 16LL * num_sms));
  k_mg_prolong<<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, x, e);
  return cudaGetLastError();
}

}  // namespace pcg

namespace pcg {

cudaError_t launch_mg_coarse_ah(const Op& fine, const Op& coarse, const double* ahf, double* ahc,
                                int num_sms, cudaStream_t s) {
  const long long g = std::max<long long>(
      1, std::min<long long>((coarse.ncols + kMgThreads - 1) / kMgThreads, 16LL * num_sms));
  k_mg_coarse_ah<<<(int)g, kMgThreads, 0, s>>>(fine, coarse, ahf, ahc);
  return cudaGetLastError();
}

}  // namespace pcg
