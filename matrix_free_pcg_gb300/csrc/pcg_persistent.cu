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
// pcg_sweeps.cuh (those of the batched kernels), separated by grid barriers.  After each barrier
// warp 0 of every block sums the per-block partials in the same fixed order
// and thread 0 takes the scalar step, so every block takes the same
// decisions (stopping test, beta, alpha) from the same numbers; block 0
// writes the history and, at the end, the device state that the host and the
// final update read.  The reductions and the scalar steps run in as few
// warps as possible: the fp64 pipe, not the issue rate, bounds them.

constexpr int kPsThreads = 512;  // 16 warps, 128 registers (the short chunks of precond_tile)
constexpr int kPsWarps = kPsThreads / 32;
// lanes of the shuffle tree over the warps' sums: a power of two >= kPsWarps
constexpr int kPsTree = kPsWarps <= 8 ? 8 : (kPsWarps <= 16 ? 16 : 32);
// A barrier wait gives up with PCG_ETIMEOUT after a second of the global
// timer, or after 2^24 polls (each an L2 round trip plus a 32 ns sleep).
constexpr long long kBarrierPolls = 1LL << 24;
constexpr unsigned long long kBarrierWaitNs = 1000000000ull;

// Block partials of NV values, in one fixed order.  Only the warps that had
// work in the sweep reduce their values with shuffles; the others contribute
// exact zeros without fp64 work (on GB300 every fp64 warp instruction holds
// the SM sub-partition's fp64 pipe for 64 cycles, so idle warps' shuffle
// trees would cost as much as busy ones').  Warp 0 adds the warp totals in a
// shuffle tree and thread 0 writes out[0..NV-1].
template <int NV>
__device__ __forceinline__ void block_partials(const double (&v)[NV], bool warp_busy,
                                               double* out) {
  __shared__ double sw[NV][kPsWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const double s = warp_busy ? warp_sum(v[j]) : 0.0;
    if (lane == 0) sw[j][w] = s;
  }
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double a = (lane < kPsWarps) ? sw[j][lane] : 0.0;
#pragma unroll
      for (int o = kPsTree / 2; o > 0; o >>= 1) a += __shfl_down_sync(0xffffffffu, a, o);
      if (lane == 0) out[j] = a;
    }
  }
}

// Grid totals of NV values from the G blocks' partials part[NV*i + j], in one
// fixed order (lane l adds the partials of blocks l, l+32, l+64, ... in turn,
// then a shuffle tree), in lane 0 of the calling warp.  Called by warp 0 of
// every block, so every block obtains the same numbers.  The loads of up to
// 8 partials per lane are issued together, ahead of the adds: one L2 round
// trip instead of one per partial.
template <int NV>
__device__ __forceinline__ void grid_totals(const double* part, int G, int lane,
                                            double (&tot)[NV]) {
  constexpr int U = 8;
#pragma unroll
  for (int j = 0; j < NV; ++j) tot[j] = 0.0;
  for (int i0 = 0; i0 < G; i0 += 32 * U) {
    double v[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + 32 * u + lane;
#pragma unroll
      for (int j = 0; j < NV; ++j) v[u][j] = (i < G) ? __ldcg(part + NV * i + j) : 0.0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int j = 0; j < NV; ++j) tot[j] += v[u][j];
    }
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) tot[j] = warp_sum(tot[j]);
}

template <bool VARY, bool RESID>
__global__ void __launch_bounds__(kPsThreads, 1) k_pcg_persistent(Op op, DevState* st,
                                                               double* __restrict__ r,
                                                               double* __restrict__ q,
                                                               double* __restrict__ z,
                                                               double* __restrict__ u,
                                                               double* __restrict__ p,
                                                               double* __restrict__ partials,
                                                               double* __restrict__ hist,
                                                               int seglen,
                                                               unsigned int absent) {
  // the scalars of Algorithm 1 live in thread 0 of each block, which takes
  // the scalar steps; the rest of the block reads alpha, beta and whether
  // the loop goes on from shared memory after a block barrier
  __shared__ double sh_alpha, sh_beta;
  __shared__ int sh_go;
  const int lane = threadIdx.x & 31;
  // warps numbered across the blocks first, so that few tiles still spread
  // over every SM of the grid (one block per SM)
  const long long warp0 = (long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const unsigned int G = gridDim.x;
  double* partM = partials;      // 2 per block: r*.r*, <r*, z>
  double* partA = partials + 2 * G;  // 1 per block: <p, q>
  const uint64_t keep = l2_keep(), stream = l2_stream();
  const long long nunits = op.ntiles * ((op.nz + seglen - 1) / seglen);
  double alpha = 0.0, beta = 0.0;
  // thread 0 only
  const double rtol = st->rtol;
  const int maxit = st->maxit;
  double kappa_old = 1.0, R0 = 0.0, R = 0.0, K = 0.0, S = 0.0;
  int it = 0, iters = 0, status = kStOK;
  bool timeout = false;
  // arrivals the grid barrier waits for; `absent` (0 in normal use) adds
  // arrivals that never come, so that a test can make the wait run out
  const unsigned int arrivals = G + absent;
  unsigned int bar_target = 0u;
  for (;;) {
    // ---- Algorithm 3 sweep
    double acc[2] = {0.0, 0.0};  // r*.r*, <r*, z>
    for (long long t = warp0; t < op.ntiles; t += nwarps)
      precond_tile<VARY, true, true>(op, t, lane, r, q, z, -alpha, keep, stream, acc[0], acc[1]);
    block_partials<2>(acc, warp0 < op.ntiles, partM + 2 * blockIdx.x);
    bar_target += arrivals;
    if (!grid_barrier(&st->bar_count, bar_target, &st->dev_error, kBarrierPolls,
                      kBarrierWaitNs)) {
      timeout = true;
      break;
    }
    if (threadIdx.x < 32) {
      double tot[2];
      grid_totals<2>(partM, G, lane, tot);
      if (lane == 0) {
        // ---- the scalar step of Algorithm 1 (as finish_precond_sweep)
        R = tot[0];
        K = tot[1];
        if (it == 0) R0 = R;
        const double ratio = (R0 > 0.0) ? sqrt(R / R0) : 0.0;
        if (blockIdx.x == 0) hist[it] = ratio;
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
          iters = it;
        } else {
          beta = K / kappa_old;
          kappa_old = K;
        }
        ++it;
        sh_beta = beta;
        sh_go = done ? 0 : 1;
      }
    }
    __syncthreads();
    if (!sh_go) break;
    beta = sh_beta;
    // ---- Algorithm 2 sweep
    double sig[1] = {0.0};
    for (long long unit = warp0; unit < nunits; unit += nwarps)
      spmv_unit<VARY, false, RESID, true>(op, unit, lane, z, r, u, p, q, alpha, beta, seglen,
                                          sig[0]);
    block_partials<1>(sig, warp0 < nunits, partA + blockIdx.x);
    bar_target += arrivals;
    if (!grid_barrier(&st->bar_count, bar_target, &st->dev_error, kBarrierPolls,
                      kBarrierWaitNs)) {
      timeout = true;
      break;
    }
    if (threadIdx.x < 32) {
      double tot[1];
      grid_totals<1>(partA, G, lane, tot);
      if (lane == 0) {
        S = tot[0];
        const bool ok = (S > 0.0) && (S < INFINITY);
        if (ok) {
          alpha = kappa_old / S;
        } else {
          alpha = 0.0;
          iters = it - 1;
          status = kStBreakdown;
        }
        sh_alpha = alpha;
        sh_go = ok ? 1 : 0;
      }
    }
    __syncthreads();
    if (!sh_go) break;
    alpha = sh_alpha;
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
  // stencil units of 8 levels: measured against 2, 4 and 16 on 128x128x64 and
  // 256x256x64 (45.96 against 46.69 us per iteration with 4, the batched
  // sweep's choice for these grids; 123.5 against 125.4 us)
  int seglen = std::min(8, op.nz);
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
