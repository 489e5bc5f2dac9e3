// Persistent solve loop of the row-tiled layout: every iteration of
// Algorithm 1 in one cooperative kernel.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 4.3 Algorithm 1 (loop), Appendix A Algorithms 2 and 3 (sweeps).
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"
#include "pcg_sweeps.cuh"

namespace pcg {
namespace {

// ------------------------------------------------ persistent solve loop
//
// For grids too small to fill the GPU, the per-launch latency of the two
// sweeps (launch, the first loads of the device scalars, the last-block
// reduction) is most of an iteration.  This kernel runs the whole loop of
// Algorithm 1 in one cooperative launch: the preconditioner sweep and the
// stencil sweep of each iteration run the tile and unit bodies of
// pcg_sweeps.cuh (those of the batched kernels), separated by grid barriers.  After each barrier every
// block sums the per-block partials in the same fixed order, so every block
// takes the same scalar decisions (stopping test, beta, alpha) from the same
// numbers; block 0 writes the history and, at the end, the device state that
// the host and the final update read.

constexpr int kPsThreads = 256;
// Polls of a barrier wait before the loop gives up with PCG_ETIMEOUT (with a
// 64 ns sleep per poll: about a second).  `absent` (0 in normal use) adds
// arrivals that never come, so that a test can make the wait run out.
constexpr long long kBarrierPolls = 1LL << 24;

// Per-block sums of two values (fixed order) into out[0], out[1].
__device__ __forceinline__ void block_partial2(double v0, double v1, double* out) {
  __shared__ double s0[kPsThreads / 32], s1[kPsThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v0 = warp_sum(v0);
  v1 = warp_sum(v1);
  if (lane == 0) {
    s0[w] = v0;
    s1[w] = v1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0, b = 0.0;
    for (int i = 0; i < kPsThreads / 32; ++i) {
      a += s0[i];
      b += s1[i];
    }
    out[0] = a;
    out[1] = b;
  }
}

// Sum of part[2*i + off], i < nparts, in one fixed order, in every thread.
__device__ __forceinline__ double grid_total(const double* part, int nparts, int off) {
  __shared__ double sh[kPsThreads / 32];
  __shared__ double tot;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double a = 0.0;
  for (int i = threadIdx.x; i < nparts; i += kPsThreads) a += __ldcg(part + 2 * i + off);
  a = warp_sum(a);
  if (lane == 0) sh[w] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int i = 0; i < kPsThreads / 32; ++i) b += sh[i];
    tot = b;
  }
  __syncthreads();
  return tot;
}

template <bool VARY, bool RESID>
__global__ void __launch_bounds__(kPsThreads) k_pcg_persistent(Op op, DevState* st,
                                                               double* __restrict__ r,
                                                               double* __restrict__ q,
                                                               double* __restrict__ z,
                                                               double* __restrict__ u,
                                                               double* __restrict__ p,
                                                               double* __restrict__ partials,
                                                               double* __restrict__ hist,
                                                               int seglen,
                                                               unsigned int absent) {
  const int lane = threadIdx.x & 31;
  // warps numbered across the blocks first, so that few tiles still spread
  // over every SM of the grid (one block per SM)
  const long long warp0 = (long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const unsigned int G = gridDim.x;
  double* partM = partials;          // 2 per block: r*.r*, <r*, z>
  double* partA = partials + 2 * G;  // 2 per block: <p, q>, unused
  const uint64_t keep = l2_keep(), stream = l2_stream();
  const double rtol = st->rtol;
  const int maxit = st->maxit;
  const long long nunits = op.ntiles * ((op.nz + seglen - 1) / seglen);
  double alpha = 0.0, beta = 0.0, kappa_old = 1.0, R0 = 0.0, R = 0.0, K = 0.0, S = 0.0;
  int it = 0, iters = 0, status = kStOK;
  bool timeout = false;
  for (;;) {
    // ---- Algorithm 3 sweep
    double accR = 0.0, accK = 0.0;
    for (long long t = warp0; t < op.ntiles; t += nwarps)
      precond_tile<VARY, true, true>(op, t, lane, r, q, z, -alpha, keep, stream, accR, accK);
    block_partial2(accR, accK, partM + 2 * blockIdx.x);
    if (!grid_barrier(&st->bar_count, &st->bar_gen, G + absent, &st->dev_error, kBarrierPolls)) {
      timeout = true;
      break;
    }
    R = grid_total(partM, G, 0);
    K = grid_total(partM, G, 1);
    // ---- the scalar step of Algorithm 1 (as finish_precond_sweep)
    if (it == 0) R0 = R;
    const double ratio = (R0 > 0.0) ? sqrt(R / R0) : 0.0;
    if (blockIdx.x == 0 && threadIdx.x == 0) hist[it] = ratio;
    bool done = true;
    if (R0 == 0.0) {
      // r_0 = 0: the initial guess solves the system
    } else if (!(R < INFINITY) || !(R0 < INFINITY)) {
      status = kStBreakdown;  // NaN or Inf in the residual
    } else if (ratio < rtol || R == 0.0) {
    } else if (it >= maxit) {
      status = (rtol > 0.0) ? kStNotConv : kStOK;
    } else if (!(K > 0.0)) {
      status = kStBreakdown;
    } else {
      done = false;
    }
    if (done) {
      iters = it++;
      break;
    }
    beta = K / kappa_old;
    kappa_old = K;
    ++it;
    // ---- Algorithm 2 sweep
    double sig = 0.0;
    for (long long unit = warp0; unit < nunits; unit += nwarps)
      spmv_unit<VARY, false, RESID, true>(op, unit, lane, z, r, u, p, q, alpha, beta, seglen,
                                          sig);
    block_partial2(sig, 0.0, partA + 2 * blockIdx.x);
    if (!grid_barrier(&st->bar_count, &st->bar_gen, G + absent, &st->dev_error, kBarrierPolls)) {
      timeout = true;
      break;
    }
    S = grid_total(partA, G, 0);
    if (!(S > 0.0) || !(S < INFINITY)) {
      alpha = 0.0;
      iters = it - 1;
      status = kStBreakdown;
      break;
    }
    alpha = kappa_old / S;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    st->alpha = alpha;
    st->beta = beta;
    st->kappa_old = kappa_old;
    st->R0 = R0;
    st->last_R = R;
    st->last_kappa = K;
    st->last_sigma = S;
    st->it = it;
    if (timeout) {
      iters = it;
      status = kStTimeout;
    }
    st->iters = iters;
    st->status = status;
    __threadfence();
    st->done = 1;
  }
}

}  // namespace

int grid_persistent(const Op& op, int num_sms) {
  int dev = 0, coop = 0;
  int occ[4] = {0, 0, 0, 0};
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[0], k_pcg_persistent<true, false>,
                                                    kPsThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[1], k_pcg_persistent<false, false>,
                                                    kPsThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[2], k_pcg_persistent<true, true>,
                                                    kPsThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[3], k_pcg_persistent<false, true>,
                                                    kPsThreads, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  // the smallest over the variants: any of them may run with this grid
  const int per_sm = std::min(std::min(occ[0], occ[1]), std::min(occ[2], occ[3]));
  if (!coop || per_sm < 1) return 0;
  long long g = (long long)per_sm * num_sms;  // every block must be resident
  // one block per tile at most: the preconditioner sweep has one tile per warp
  // and the warps are spread over the blocks first
  g = std::min(g, op.ntiles);
  return (int)std::max<long long>(g, 1);
}

cudaError_t launch_persistent(const Op& op, DevState* st, double* r, double* q, double* z,
                              double* u, double* p, double* partials, double* hist, int grid,
                              unsigned int absent, cudaStream_t s) {
  Op o = op;
  int seglen = tiled_spmv_seglen(op, grid);
  void* args[] = {&o, &st, &r, &q, &z, &u, &p, &partials, &hist, &seglen, &absent};
  const void* fn;
  if (op.varying)
    fn = op.az_resid ? reinterpret_cast<const void*>(k_pcg_persistent<true, true>)
                     : reinterpret_cast<const void*>(k_pcg_persistent<true, false>);
  else
    fn = op.az_resid ? reinterpret_cast<const void*>(k_pcg_persistent<false, true>)
                     : reinterpret_cast<const void*>(k_pcg_persistent<false, false>);
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kPsThreads), args, 0, s);
}

}  // namespace pcg
