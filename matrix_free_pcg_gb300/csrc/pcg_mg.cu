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
//   k_mg_first     x = omega M^{-1} b (on the finest level fused with the
//                  residual update r <- r - alpha q of Algorithm 3 and ||r||^2)
//   k_mg_smooth    further smoothing steps (nu > 1)
//   k_mg_restrict  b_{l+1} = R (b - A x)
//   ... the coarser levels ...
//   k_mg_prolong   x += P x_{l+1}
//   k_mg_smooth    nu smoothing steps (on the finest level the last one also
//                  reduces <r, z> and takes the scalar step of Algorithm 1)
#include <algorithm>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"
#include "pcg_sweeps.cuh"

namespace pcg {
namespace {

constexpr int kMgThreads = 256;  // restriction and prolongation blocks

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

// x = omega M^{-1} b, one warp per tile of 32 columns (the Thomas tile body
// of the preconditioner sweep).  FUSED: b <- b - alpha q first, and ||b||^2
// reduced into st->mg_R.
template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTmThreads) k_mg_first(Op op, DevState* st,
                                                         double* __restrict__ b,
                                                         const double* __restrict__ q,
                                                         double* __restrict__ x, double omega,
                                                         double* __restrict__ partials) {
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
    if (grid_sum2<kTmThreads>(accR, 0.0, partials, &st->ticket_m, R, unused)) st->mg_R = R;
  }
}

// xout = xin + omega M^{-1} (b - A xin), one warp per tile, one thread per
// column walking up (residual and forward elimination, w kept in xout) and
// down (back substitution).  FUSED: <b, xout> reduced, then the scalar step
// of Algorithm 1 with ||r||^2 from st->mg_R.
template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTmThreads) k_mg_smooth(Op op, DevState* st,
                                                          const double* __restrict__ b,
                                                          const double* __restrict__ xin,
                                                          double* __restrict__ xout,
                                                          double omega,
                                                          double* __restrict__ partials,
                                                          double* __restrict__ hist) {
  if (ld_done(st)) return;
  const int nz = op.nz;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint64_t keep = l2_keep(), stream = l2_stream();
  const int fs = VARY ? kTile : 1;  // factor stride between levels
  double accK = 0.0;
  for (long long t = warp0; t < op.ntiles; t += nwarps) {
    const long long col = t * kTile + lane;
    if (col >= op.ncols) continue;
    const long long base = t * nz * kTile + lane;
    const Nbr nb = neighbours(op, col);
    const long long bE = tiled_base(nb.e, nz), bW = tiled_base(nb.w, nz);
    const long long bN = tiled_base(nb.n, nz), bS = tiled_base(nb.s, nz);
    const double* __restrict__ fi = VARY ? op.tinvd + base : op.lev + LV_INVD * nz;
    const double* __restrict__ fn = VARY ? op.tnphi + base : op.lev + LV_NPHI * nz;
    double xd = 0.0, xc = xin[base], y = 0.0, nprev = 0.0, w = 0.0;
#pragma unroll 2
    for (int k = 0; k < nz; ++k) {
      const long long ko = (long long)k * kTile, o = base + ko;
      const double xu = (k + 1 < nz) ? xin[o + kTile] : 0.0;
      const double s = b[o] - stencil_at<VARY>(op, xin, o, ko, k, bE, bW, bN, bS, xd, xc, xu);
      y = fma(nprev, y, s);
      w = y * (VARY ? ld_hint(fi + k * fs, stream) : __ldg(fi + k));
      st_hint(xout + o, w, keep);
      nprev = VARY ? ld_hint(fn + k * fs, keep) : __ldg(fn + k);
      xd = xc;
      xc = xu;
    }
    double zz = w;
    for (int k = nz - 1; k >= 0; --k) {
      const long long o = base + (long long)k * kTile;
      if (k < nz - 1)
        zz = fma(VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k), zz, ld_hint(xout + o, stream));
      const double out = fma(omega, zz, xin[o]);
      st_hint(xout + o, out, stream);
      if (FUSED) accK = fma(b[o], out, accK);
    }
  }
  if (FUSED) {
    double K, unused;
    if (grid_sum2<kTmThreads>(accK, 0.0, partials, &st->ticket_m, K, unused))
      finish_precond_sweep(st, st->mg_R, K, hist);
  }
}

// bc = R (b - A x): one thread per coarse column (I, J); per layer, the
// residuals of the fine columns (2I, 2J), (2I+1, 2J), (2I, 2J+1),
// (2I+1, 2J+1) summed in that order.
template <bool VARY>
__global__ void __launch_bounds__(kMgThreads) k_mg_restrict(Op f, Op c, const DevState* st,
                                                            const double* __restrict__ b,
                                                            const double* __restrict__ x,
                                                            double* __restrict__ bc) {
  if (ld_done(st)) return;
  const int nz = f.nz;
  for (long long C = blockIdx.x * (long long)blockDim.x + threadIdx.x; C < c.ncols;
       C += (long long)gridDim.x * blockDim.x) {
    const long long J = C / c.nx;
    const int I = (int)(C - J * c.nx);
    long long base[4], bE[4], bW[4], bN[4], bS[4];
    double xd[4], xc[4];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const long long col = (2 * J + (qd >> 1)) * f.nx + 2 * I + (qd & 1);
      const Nbr nb = neighbours(f, col);
      base[qd] = tiled_base(col, nz);
      bE[qd] = tiled_base(nb.e, nz);
      bW[qd] = tiled_base(nb.w, nz);
      bN[qd] = tiled_base(nb.n, nz);
      bS[qd] = tiled_base(nb.s, nz);
      xd[qd] = 0.0;
      xc[qd] = x[base[qd]];
    }
    const long long cb = tiled_base(C, nz);
    for (int k = 0; k < nz; ++k) {
      const long long ko = (long long)k * kTile;
      double t[4];
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        const long long o = base[qd] + ko;
        const double xu = (k + 1 < nz) ? x[o + kTile] : 0.0;
        t[qd] = b[o] - stencil_at<VARY>(f, x, o, ko, k, bE[qd], bW[qd], bN[qd], bS[qd], xd[qd],
                                        xc[qd], xu);
        xd[qd] = xc[qd];
        xc[qd] = xu;
      }
      bc[cb + ko] = ((t[0] + t[1]) + t[2]) + t[3];
    }
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
  const int cap = 16 / kTmWarpsPerBlock;  // 16 warps per SM: the w of their tiles stay in L2
  return op.varying ? occupancy_grid(k_mg_smooth<true, true>, kTmThreads, cap, work, num_sms)
                    : occupancy_grid(k_mg_smooth<false, true>, kTmThreads, cap, work, num_sms);
}

cudaError_t launch_mg_first(const Op& op, DevState* st, double* b, const double* q, double* x,
                            double omega, bool fused, double* partials, int grid,
                            cudaStream_t s) {
  if (op.varying) {
    if (fused)
      k_mg_first<true, true><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials);
    else
      k_mg_first<true, false><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials);
  } else {
    if (fused)
      k_mg_first<false, true><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials);
    else
      k_mg_first<false, false><<<grid, kTmThreads, 0, s>>>(op, st, b, q, x, omega, partials);
  }
  return cudaGetLastError();
}

cudaError_t launch_mg_smooth(const Op& op, DevState* st, const double* b, const double* xin,
                             double* xout, double omega, bool fused, double* partials,
                             double* hist, int grid, cudaStream_t s) {
  if (op.varying) {
    if (fused)
      k_mg_smooth<true, true><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega, partials,
                                                          hist);
    else
      k_mg_smooth<true, false><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega, partials,
                                                           hist);
  } else {
    if (fused)
      k_mg_smooth<false, true><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega, partials,
                                                           hist);
    else
      k_mg_smooth<false, false><<<grid, kTmThreads, 0, s>>>(op, st, b, xin, xout, omega,
                                                            partials, hist);
  }
  return cudaGetLastError();
}

cudaError_t launch_mg_restrict(const Op& fine, const Op& coarse, const DevState* st,
                               const double* b, const double* x, double* bc, int num_sms,
                               cudaStream_t s) {
  const long long g = std::max<long long>(
      1, std::min<long long>((coarse.ncols + kMgThreads - 1) / kMgThreads, 8LL * num_sms));
  if (fine.varying)
    k_mg_restrict<true><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, bc);
  else
    k_mg_restrict<false><<<(int)g, kMgThreads, 0, s>>>(fine, coarse, st, b, x, bc);
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
