// Row-tiled solver layout: the paper's eq. (22) ordering (horizontal index
// fastest) in blocked form, with its two fused sweeps (stored or rebuilt
// factors), the conversions from and to the caller's layout, and the
// persistent loop that runs every iteration of a small grid in one kernel.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 6.1, eq. (22) (layout), section 4.3 Algorithm 1 (loop), Appendix A
// Algorithms 2 and 3 (sweeps).
//
// Cell (column c, level k) sits at (c/32 * nz + k) * 32 + c%32: level-major
// within tiles of 32 consecutive columns, so it works for any nx.  A warp
// owns a tile, one lane per column, and every level of the tile is one
// 256-byte line: the preconditioner needs no shared memory at all and keeps
// w in z, and the stencil walks its column with a register window along k.
// The caller's b and x stay column-contiguous; they are converted at the
// start and the end of a solve.  Vectors in this layout hold ntiles*32*nz
// values (the last tile padded to 32 columns; padded lanes never compute).
#include <algorithm>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"
#include "pcg_sweeps.cuh"

namespace pcg {
namespace {

// Column-contiguous <-> row-tiled conversion, 32 columns x 32 levels per
// block through a padded shared tile (coalesced on both sides).
// TO_TILED: dst_t = src_k.  Otherwise dst_k = src_t + alpha * p_t (AXPY,
// alpha from the device state: the deferred x += alpha p of Algorithm 1), or
// a plain copy.  With alpha = 0 -- a solve that stopped before its first
// direction, or a breakdown that keeps the iterate before the current one --
// dst_k = src_t and p_t is not read: the batched row-tiled start leaves p
// unwritten, so it may hold anything (a NaN would survive 0 * p).
template <bool TO_TILED, bool AXPY>
__global__ void __launch_bounds__(256) k_retile(Op op, const DevState* st,
                                                const double* __restrict__ src,
                                                const double* __restrict__ pt,
                                                double* __restrict__ dst) {
  __shared__ double tile[kTile][kTile + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int nz = op.nz;
  const long long t = blockIdx.x;
  const int k0 = blockIdx.y * kTile;
  const long long col0 = t * kTile;
  const int nc = (int)min((long long)kTile, op.ncols - col0);
  const int nk = min(kTile, nz - k0);
  const double alpha = AXPY ? st->alpha : 0.0;
  const bool axpy = AXPY && alpha != 0.0;
  if (TO_TILED) {
    for (int c = ty; c < nc; c += 8)
      if (tx < nk) tile[c][tx] = src[(col0 + c) * nz + k0 + tx];
    __syncthreads();
    for (int k = ty; k < nk; k += 8)
      if (tx < nc) {
        dst[(t * nz + k0 + k) * kTile + tx] = tile[tx][k];
      }
  } else {
    for (int k = ty; k < nk; k += 8)
      if (tx < nc) {
        const long long o = (t * nz + k0 + k) * kTile + tx;
        tile[tx][k] = axpy ? fma(alpha, pt[o], src[o]) : src[o];
      }
    __syncthreads();
    for (int c = ty; c < nc; c += 8)
      if (tx < nk) dst[(col0 + c) * nz + k0 + tx] = tile[c][tx];
  }
}

// Algorithm 3 sweep (FUSED: r* = r - alpha q, then z = M^{-1} r*, with the
// partial sums of r*.r* and <r*, z>) or plain z = M^{-1} r, on row-tiled
// vectors.  One warp per tile, one lane per column.
//
// Every load is independent of the recurrences, so the sweep fetches the
// operands of kTmChunk levels (r, q and the two Thomas factors forward; w and
// nphi backward) one chunk ahead into registers: the loads of chunk c+1 are
// in flight while chunk c computes.  w is written into z on the way up with
// the L2 evict-last hint and replaced by z on the way down; streamed data
// carries evict-first.  FIRST: the first sweep of a solve (see precond_tile).
template <bool VARY, bool FUSED, bool FIRST = false>
__global__ void __launch_bounds__(kTmThreads) k_precond_tiled(Op op, DevState* st,
                                                              double* __restrict__ r,
                                                              const double* __restrict__ q,
                                                              double* __restrict__ z,
                                                              double* __restrict__ partials,
                                                              double* __restrict__ hist) {
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const double nalpha = FUSED ? -st->alpha : 0.0;
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accR = 0.0, accK = 0.0;
  for (long long t = warp0; t < op.ntiles; t += nwarps)
    precond_tile<VARY, FUSED, false, false, FIRST>(op, t, lane, r, q, z, nalpha, keep, stream,
                                                   accR, accK);
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTmThreads>(accR, accK, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

// Algorithm 3 sweep with the factors rebuilt in the sweep (a_h per column),
// as the paper's Algorithm 3 does, instead of read from per-cell arrays:
//   diag_k = (h_k mass + T_{k+1/2} + T_{k-1/2}) + h_k * (sum of the four faces)
//   D_k = diag_k - T_{k-1/2} * (T_{k-1/2}/D_{k-1}),   1/D_k,   T_{k+1/2}/D_k,
// each rounded like the set-up kernels round them (no contraction), so the
// sweep gives bit for bit the result of the stored-factor sweep.  This
// trades 16 bytes per cell of factor reads for a division, a reciprocal and
// four more fp64 operations per cell.  T_{k+1/2}/D_k, needed again by the
// back substitution, goes to a per-warp scratch region (32 x nz doubles,
// level-major) that stays in L2 like w.
template <bool FUSED>
__global__ void __launch_bounds__(kTmThreads) k_precond_tiled_rc(Op op, DevState* st,
                                                                 double* __restrict__ r,
                                                                 const double* __restrict__ q,
                                                                 double* __restrict__ z,
                                                                 double* __restrict__ partials,
                                                                 double* __restrict__ hist) {
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  double* __restrict__ ns = op.nscratch + warp0 * nz * kTile + lane;  // level k at ns[k*32]
  const double nalpha = FUSED ? -st->alpha : 0.0;
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accR = 0.0, accK = 0.0;
  for (long long t = warp0; t < op.ntiles; t += nwarps) {
    const long long col = t * kTile + lane;
    if (col >= op.ncols) continue;
    const long long base = t * nz * kTile + lane;
    double* __restrict__ rt = r + base;
    const double* __restrict__ qt = FUSED ? q + base : nullptr;
    double* __restrict__ zt = z + base;
    const Nbr nb = neighbours(op, col);
    const double sf = op.faceE[col] + op.faceE[nb.w] + op.faceN[col] + op.faceN[nb.s];
    // ---- forward
    double cr[kTmChunk], cq[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const bool in = j < nz;
      cr[j] = in ? ld_hint(rt + j * kTile, stream) : 0.0;
      cq[j] = (FUSED && in) ? ld_hint(qt + j * kTile, stream) : 0.0;
    }
    double y = 0.0, nprev = 0.0, w = 0.0;
#pragma unroll 1
    for (int k0 = 0; k0 < nz; k0 += kTmChunk) {
      double nr[kTmChunk], nq[kTmChunk];
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        const int k = k0 + kTmChunk + j;
        const bool in = k < nz;
        nr[j] = in ? ld_hint(rt + k * kTile, stream) : 0.0;
        nq[j] = (FUSED && in) ? ld_hint(qt + k * kTile, stream) : 0.0;
      }
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        const int k = k0 + j;
        if (k < nz) {
          const double diag = __dadd_rn(__ldg(lev + LV_DIAG * nz + k),
                                        __dmul_rn(__ldg(lev + LV_H * nz + k), sf));
          const double D = __dsub_rn(diag, __dmul_rn(__ldg(lev + LV_TDN * nz + k), nprev));
          const double invd = 1.0 / D;
          const double nphi = __ldg(lev + LV_TUP * nz + k) / D;
          double rk = cr[j];
          if (FUSED) {
            rk = fma(nalpha, cq[j], rk);
            accR = fma(rk, rk, accR);
            st_hint(rt + k * kTile, rk, stream);
          }
          y = fma(nprev, y, rk);
          w = y * invd;
          if (FUSED) accK = fma(y, w, accK);
          st_hint(zt + k * kTile, w, keep);
          st_hint(ns + k * kTile, nphi, keep);
          nprev = nphi;
        }
      }
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        cr[j] = nr[j];
        cq[j] = nq[j];
      }
    }
    // ---- backward, as in the stored-factor sweep with nphi from the scratch
    double zz = w;
    double bw[kTmChunk], bn[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = nz - 2 - j;
      bw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
      bn[j] = (k >= 0) ? ld_hint(ns + k * kTile, stream) : 0.0;
    }
#pragma unroll 1
    for (int kb = nz - 2; kb >= 0; kb -= kTmChunk) {
      double nw[kTmChunk], nb2[kTmChunk];
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        const int k = kb - kTmChunk - j;
        nw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
        nb2[j] = (k >= 0) ? ld_hint(ns + k * kTile, stream) : 0.0;
      }
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        const int k = kb - j;
        if (k >= 0) {
          zz = fma(bn[j], zz, bw[j]);
          st_hint(zt + k * kTile, zz, stream);
        }
      }
#pragma unroll
      for (int j = 0; j < kTmChunk; ++j) {
        bw[j] = nw[j];
        bn[j] = nb2[j];
      }
    }
  }
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTmThreads>(accR, accK, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

// Algorithm 2 sweep on row-tiled vectors: u += alpha p; p = z + beta p;
// q = A z + beta q; <p,q>.  One thread per column walking up the levels
// with z_{k-1}, z_k, z_{k+1} in registers (RESID: A z = r + (A - M) z, no
// vertical terms); the horizontal neighbours are fixed offsets from the
// column's own.  The unit of work is a segment of
// seglen levels of one tile (the stencil has no recurrence along k), so that
// grids with few tiles still give every warp several units; units are
// assigned statically (segment-major), which keeps the sum bitwise
// repeatable.  FIRST: the first sweep of a solve (see spmv_unit).
template <bool VARY, bool RECOMP, bool RESID, bool FIRST = false>
__global__ void __launch_bounds__(256) k_spmv_tiled(Op op, DevState* st,
                                                    const double* __restrict__ z,
                                                    const double* __restrict__ r,
                                                    double* __restrict__ u,
                                                    double* __restrict__ p,
                                                    double* __restrict__ q,
                                                    double* __restrict__ partials,
                                                    int seglen) {
  if (ld_done(st)) return;
  const double alpha = st->alpha, beta = st->beta;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  double sig = 0.0;
  const long long nunits = op.ntiles * ((op.nz + seglen - 1) / seglen);
  for (long long unit = warp0; unit < nunits; unit += nwarps)
    spmv_unit<VARY, RECOMP, RESID, false, FIRST>(op, unit, lane, z, r, u, p, q, alpha, beta,
                                                 seglen, sig);
  double S, unused;
  if (grid_sum2<256>(sig, 0.0, partials, &st->ticket_a, S, unused)) {
    st->last_sigma = S;
    if (!(S > 0.0) || !(S < INFINITY)) {
      st->alpha = 0.0;
      st->iters = st->it - 1;
      st->status = kStBreakdown;
      __threadfence();
      st->done = 1;
    } else {
      st->alpha = st->kappa_old / S;
    }
  }
}

}  // namespace

cudaError_t launch_to_tiled(const Op& op, const double* src_k, double* dst_t, cudaStream_t s) {
  dim3 g((unsigned)op.ntiles, (unsigned)((op.nz + kTile - 1) / kTile));
  k_retile<true, false><<<g, 256, 0, s>>>(op, nullptr, src_k, nullptr, dst_t);
  return cudaGetLastError();
}

cudaError_t launch_from_tiled(const Op& op, const DevState* st, const double* src_t,
                              const double* p_t, double* dst_k, cudaStream_t s) {
  dim3 g((unsigned)op.ntiles, (unsigned)((op.nz + kTile - 1) / kTile));
  if (p_t)
    k_retile<false, true><<<g, 256, 0, s>>>(op, st, src_t, p_t, dst_k);
  else
    k_retile<false, false><<<g, 256, 0, s>>>(op, st, src_t, nullptr, dst_k);
  return cudaGetLastError();
}

cudaError_t launch_precond_tiled(const Op& op, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s, bool first) {
  if (first && !op.recompute) {
    if (op.varying)
      k_precond_tiled<true, true, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
    else
      k_precond_tiled<false, true, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials,
                                                                      hist);
    return cudaGetLastError();
  }
  if (op.varying && op.recompute)
    k_precond_tiled_rc<true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  else if (op.varying)
    k_precond_tiled<true, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  else
    k_precond_tiled<false, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  return cudaGetLastError();
}

cudaError_t launch_spmv_tiled(const Op& op, DevState* st, const double* z, const double* r,
                              double* u, double* p, double* q, double* partials, int grid,
                              cudaStream_t s, bool first) {
  const int seglen = tiled_spmv_seglen(op, grid);
  const bool rs = op.az_resid != 0;
  if (first && !op.recompute) {
    if (op.varying) {
      if (rs)
        k_spmv_tiled<true, false, true, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                                   seglen);
      else
        k_spmv_tiled<true, false, false, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                                    seglen);
    } else {
      if (rs)
        k_spmv_tiled<false, false, true, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                                    seglen);
      else
        k_spmv_tiled<false, false, false, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q,
                                                                     partials, seglen);
    }
    return cudaGetLastError();
  }
  if (op.varying && op.recompute) {
    if (rs)
      k_spmv_tiled<true, true, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials, seglen);
    else
      k_spmv_tiled<true, true, false><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials, seglen);
  } else if (op.varying) {
    if (rs)
      k_spmv_tiled<true, false, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials, seglen);
    else
      k_spmv_tiled<true, false, false><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                             seglen);
  } else {
    if (rs)
      k_spmv_tiled<false, false, true><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                             seglen);
    else
      k_spmv_tiled<false, false, false><<<grid, 256, 0, s>>>(op, st, z, r, u, p, q, partials,
                                                              seglen);
  }
  return cudaGetLastError();
}

int grid_tiled_precond(const Op& op, int num_sms) {
  int a = 0;
  if (op.varying)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_precond_tiled<true, true>, kTmThreads, 0);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_precond_tiled<false, true>, kTmThreads, 0);
  const int per_sm = std::max(1, std::min(a, kTmWarpsPerSm / (kTmThreads / 32)));
  long long g = (long long)per_sm * num_sms;
  const long long work = (op.ntiles + kTmThreads / 32 - 1) / (kTmThreads / 32);
  if (g > work) g = work;
  return (int)(g < 1 ? 1 : g);
}

int grid_tiled_spmv(const Op& op, int num_sms) {
  int b = 0;
  if (op.varying)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_spmv_tiled<true, false, false>, 256, 0);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_spmv_tiled<false, false, false>, 256, 0);
  long long g = (long long)std::max(1, b) * num_sms;
  // enough blocks for one unit per warp at the shortest segments
  const long long units = op.ntiles * std::max(1, op.nz / 4);
  const long long work = (units + 7) / 8;  // 8 warps per block
  if (g > work) g = work;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace pcg
