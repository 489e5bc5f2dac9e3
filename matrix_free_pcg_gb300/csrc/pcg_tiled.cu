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

namespace pcg {
namespace {

// Preconditioner sweep: threads per block and levels per register chunk.
constexpr int kTmThreads = kTmWarpsPerBlock * 32;
constexpr int kTmChunk = 8;

__device__ __forceinline__ long long tiled_base(long long col, int nz) {
  return (col >> 5) * (long long)nz * kTile + (col & 31);
}

// Column-contiguous <-> row-tiled conversion, 32 columns x 32 levels per
// block through a padded shared tile (coalesced on both sides).
// TO_TILED: dst_t = src_k.  Otherwise dst_k = src_t + alpha * p_t (AXPY,
// alpha from the device state: the deferred x += alpha p of Algorithm 1), or
// a plain copy.
// With TO_TILED, zero1/zero2 (may be NULL) are cleared at the same row-tiled
// positions (p and q at the start of a solve).
template <bool TO_TILED, bool AXPY>
__global__ void __launch_bounds__(256) k_retile(Op op, const DevState* st,
                                                const double* __restrict__ src,
                                                const double* __restrict__ pt,
                                                double* __restrict__ dst,
                                                double* __restrict__ zero1,
                                                double* __restrict__ zero2) {
  __shared__ double tile[kTile][kTile + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int nz = op.nz;
  const long long t = blockIdx.x;
  const int k0 = blockIdx.y * kTile;
  const long long col0 = t * kTile;
  const int nc = (int)min((long long)kTile, op.ncols - col0);
  const int nk = min(kTile, nz - k0);
  const double alpha = AXPY ? st->alpha : 0.0;
  if (TO_TILED) {
    for (int c = ty; c < nc; c += 8)
      if (tx < nk) tile[c][tx] = src[(col0 + c) * nz + k0 + tx];
    __syncthreads();
    for (int k = ty; k < nk; k += 8)
      if (tx < nc) {
        const long long o = (t * nz + k0 + k) * kTile + tx;
        dst[o] = tile[tx][k];
        if (zero1) zero1[o] = 0.0;
        if (zero2) zero2[o] = 0.0;
      }
  } else {
    for (int k = ty; k < nk; k += 8)
      if (tx < nc) {
        const long long o = (t * nz + k0 + k) * kTile + tx;
        tile[tx][k] = AXPY ? fma(alpha, pt[o], src[o]) : src[o];
      }
    __syncthreads();
    for (int c = ty; c < nc; c += 8)
      if (tx < nk) dst[(col0 + c) * nz + k0 + tx] = tile[c][tx];
  }
}

// One tile of the preconditioner sweep (see k_precond_tiled), for the lane's
// column: accumulates r*.r* and <r*, z> into accR, accK (FUSED).  COHERENT:
// q was written by other blocks of the same launch (the persistent loop), so
// it is read from L2, past the SM's non-coherent L1.
template <bool VARY, bool FUSED, bool COHERENT = false>
__device__ __forceinline__ void precond_tile(const Op& op, long long t, int lane,
                                             double* __restrict__ r, const double* __restrict__ q,
                                             double* __restrict__ z, double nalpha, uint64_t keep,
                                             uint64_t stream, double& accR, double& accK) {
  const int nz = op.nz;
  const int fs = VARY ? kTile : 1;  // factor stride between levels
  if (t * kTile + lane >= op.ncols) return;
  const long long base = t * nz * kTile + lane;
  double* __restrict__ rt = r + base;
  const double* __restrict__ qt = FUSED ? q + base : nullptr;
  double* __restrict__ zt = z + base;
  const double* __restrict__ fi = VARY ? op.tinvd + base : op.lev + LV_INVD * nz;
  const double* __restrict__ fn = VARY ? op.tnphi + base : op.lev + LV_NPHI * nz;
  // ---- forward: level k uses nphi_{k-1} (0 at k = 0) and 1/D_k
  double cr[kTmChunk], cq[kTmChunk], ci[kTmChunk], cn[kTmChunk];
#pragma unroll
  for (int j = 0; j < kTmChunk; ++j) {
    const bool in = j < nz;
    cr[j] = in ? ld_hint(rt + j * kTile, stream) : 0.0;
    cq[j] = (FUSED && in) ? (COHERENT ? __ldcg(qt + j * kTile) : ld_hint(qt + j * kTile, stream))
                          : 0.0;
    ci[j] = in ? (VARY ? ld_hint(fi + j * fs, stream) : __ldg(fi + j)) : 0.0;
    cn[j] = in ? (VARY ? ld_hint(fn + j * fs, keep) : __ldg(fn + j)) : 0.0;
  }
  double y = 0.0, nprev = 0.0, w = 0.0;
#pragma unroll 1
  for (int k0 = 0; k0 < nz; k0 += kTmChunk) {
    double nr[kTmChunk], nq[kTmChunk], ni[kTmChunk], nn[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = k0 + kTmChunk + j;
      const bool in = k < nz;
      nr[j] = in ? ld_hint(rt + k * kTile, stream) : 0.0;
      nq[j] = (FUSED && in) ? (COHERENT ? __ldcg(qt + k * kTile) : ld_hint(qt + k * kTile, stream))
                            : 0.0;
      ni[j] = in ? (VARY ? ld_hint(fi + k * fs, stream) : __ldg(fi + k)) : 0.0;
      nn[j] = in ? (VARY ? ld_hint(fn + k * fs, keep) : __ldg(fn + k)) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = k0 + j;
      if (k < nz) {
        double rk = cr[j];
        if (FUSED) {
          rk = fma(nalpha, cq[j], rk);
          accR = fma(rk, rk, accR);
          st_hint(rt + k * kTile, rk, stream);
        }
        y = fma(nprev, y, rk);
        w = y * ci[j];
        if (FUSED) accK = fma(y, w, accK);
        st_hint(zt + k * kTile, w, keep);
        nprev = cn[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      cr[j] = nr[j];
      cq[j] = nq[j];
      ci[j] = ni[j];
      cn[j] = nn[j];
    }
  }
  // ---- backward: z_{nz-1} = w_{nz-1} (in place); level k uses nphi_k.
  // Chunk b holds levels kb, kb-1, ..., kb-kTmChunk+1 with kb = nz-2-b*kTmChunk.
  double zz = w;
  double bw[kTmChunk], bn[kTmChunk];
#pragma unroll
  for (int j = 0; j < kTmChunk; ++j) {
    const int k = nz - 2 - j;
    bw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
    bn[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
  }
#pragma unroll 1
  for (int kb = nz - 2; kb >= 0; kb -= kTmChunk) {
    double nw[kTmChunk], nb[kTmChunk];
#pragma unroll
    for (int j = 0; j < kTmChunk; ++j) {
      const int k = kb - kTmChunk - j;
      nw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
      nb[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
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
      bn[j] = nb[j];
    }
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
// carries evict-first.
template <bool VARY, bool FUSED>
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
    precond_tile<VARY, FUSED>(op, t, lane, r, q, z, nalpha, keep, stream, accR, accK);
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

// One unit (a segment of seglen levels of one tile) of the stencil sweep (see
// k_spmv_tiled) for the lane's column; accumulates <p, q> into sig.
// COHERENT: z was written by other blocks of the same launch (the persistent
// loop), so it is read from L2, past the SM's non-coherent L1.
template <bool VARY, bool RECOMP, bool COHERENT = false>
__device__ __forceinline__ void spmv_unit(const Op& op, long long unit, int lane,
                                          const double* __restrict__ z, double* __restrict__ u,
                                          double* __restrict__ p, double* __restrict__ q,
                                          double alpha, double beta, int seglen, double& sig) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const long long t = unit % op.ntiles;
  const int k0 = (int)(unit / op.ntiles) * seglen;
  const int k1 = min(nz, k0 + seglen);
  const long long col = t * kTile + lane;
  if (col >= op.ncols) return;
  const long long base = t * nz * kTile + lane;
  const Nbr nb = neighbours(op, col);
  const long long bE = tiled_base(nb.e, nz), bW = tiled_base(nb.w, nz);
  const long long bN = tiled_base(nb.n, nz), bS = tiled_base(nb.s, nz);
  double aE = 0.0, aW = 0.0, aN = 0.0, aS = 0.0;
  if (RECOMP) {
    aE = __ldg(op.faceE + col);
    aW = __ldg(op.faceE + nb.w);
    aN = __ldg(op.faceN + col);
    aS = __ldg(op.faceN + nb.s);
  }
  // RECOMP: the diagonal rebuilt as the set-up kernel rounds it
  const double sf = RECOMP ? aE + aW + aN + aS : 0.0;
  auto ldz = [&](long long o) { return COHERENT ? __ldcg(z + o) : z[o]; };
  double zd = (k0 > 0) ? ldz(base + (long long)(k0 - 1) * kTile) : 0.0;
  double zc = ldz(base + (long long)k0 * kTile);
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    const long long o = base + (long long)k * kTile;
    const long long ko = (long long)k * kTile;
    const double zu = (k + 1 < nz) ? ldz(o + kTile) : 0.0;
    const double zE = ldz(bE + ko), zW = ldz(bW + ko), zN = ldz(bN + ko), zS = ldz(bS + ko);
    double uc = __ldcs(u + o);
    double pc = __ldcs(p + o);
    const double qc = __ldcs(q + o);
    uc = fma(alpha, pc, uc);
    pc = fma(beta, pc, zc);
    double a;
    if (VARY) {
      // per-cell horizontal weights -h_k a_f (west and south: the
      // neighbours' east and north weights), rebuilt with the set-up's
      // rounding under RECOMP
      double d, cE, cW, cN, cS;
      if (RECOMP) {
        const double hw = __ldg(lev + LV_HW * nz + k);
        d = __dadd_rn(__ldg(lev + LV_DIAG * nz + k), __dmul_rn(__ldg(lev + LV_H * nz + k), sf));
        cE = __dmul_rn(hw, aE);
        cW = __dmul_rn(hw, aW);
        cN = __dmul_rn(hw, aN);
        cS = __dmul_rn(hw, aS);
      } else {
        d = __ldcs(op.cdiag_t + o);
        cE = __ldg(op.cwE_t + o);
        cW = __ldg(op.cwE_t + bW + ko);
        cN = __ldg(op.cwN_t + o);
        cS = __ldg(op.cwN_t + bS + ko);
      }
      a = fma(d, zc, beta * qc);
      a = fma(__ldg(lev + LV_UP * nz + k), zu, a);
      a = fma(__ldg(lev + LV_DN * nz + k), zd, a);
      a = fma(cE, zE, a);
      a = fma(cW, zW, a);
      a = fma(cN, zN, a);
      a = fma(cS, zS, a);
    } else {
      const double hs = (zE + zW) + (zN + zS);
      a = fma(__ldg(lev + LV_DIAG * nz + k), zc, beta * qc);
      a = fma(__ldg(lev + LV_UP * nz + k), zu, a);
      a = fma(__ldg(lev + LV_DN * nz + k), zd, a);
      a = fma(__ldg(lev + LV_HW * nz + k), hs, a);
    }
    sig = fma(pc, a, sig);
    __stcs(u + o, uc);
    __stcs(p + o, pc);
    __stcs(q + o, a);
    zd = zc;
    zc = zu;
  }
}

// Algorithm 2 sweep on row-tiled vectors: u += alpha p; p = z + beta p;
// q = A z + beta q; <p,q>.  One thread per column walking up the levels
// with z_{k-1}, z_k, z_{k+1} in registers; the horizontal neighbours are
// fixed offsets from the column's own.  The unit of work is a segment of
// seglen levels of one tile (the stencil has no recurrence along k), so that
// grids with few tiles still give every warp several units; units are
// assigned statically (segment-major), which keeps the sum bitwise
// repeatable.
template <bool VARY, bool RECOMP>
__global__ void __launch_bounds__(256) k_spmv_tiled(Op op, DevState* st,
                                                    const double* __restrict__ z,
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
    spmv_unit<VARY, RECOMP>(op, unit, lane, z, u, p, q, alpha, beta, seglen, sig);
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

// ------------------------------------------------ persistent solve loop
//
// For grids too small to fill the GPU, the per-launch latency of the two
// sweeps (launch, the first loads of the device scalars, the last-block
// reduction) is most of an iteration.  This kernel runs the whole loop of
// Algorithm 1 in one cooperative launch: the preconditioner sweep and the
// stencil sweep of each iteration are the same tile and unit bodies as the
// two kernels above, separated by grid barriers.  After each barrier every
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

template <bool VARY>
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
      spmv_unit<VARY, false, true>(op, unit, lane, z, u, p, q, alpha, beta, seglen, sig);
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

// Levels per work unit of the tiled stencil sweep: whole columns when there
// are at least 8 tiles per resident warp, else segments short enough to give
// every warp about 8 units (at least 4 levels each).
int tiled_spmv_seglen(const Op& op, int grid) {
  const long long warps = (long long)grid * 8;
  const long long want = 8 * warps;
  if (op.ntiles >= want || op.nz <= 4) return op.nz;
  long long nseg = (want + op.ntiles - 1) / op.ntiles;
  nseg = std::min<long long>(nseg, op.nz / 4);
  return (int)((op.nz + nseg - 1) / nseg);
}

}  // namespace

cudaError_t launch_to_tiled(const Op& op, const double* src_k, double* dst_t, cudaStream_t s,
                            double* zero1, double* zero2) {
  dim3 g((unsigned)op.ntiles, (unsigned)((op.nz + kTile - 1) / kTile));
  k_retile<true, false><<<g, 256, 0, s>>>(op, nullptr, src_k, nullptr, dst_t, zero1, zero2);
  return cudaGetLastError();
}

cudaError_t launch_from_tiled(const Op& op, const DevState* st, const double* src_t,
                              const double* p_t, double* dst_k, cudaStream_t s) {
  dim3 g((unsigned)op.ntiles, (unsigned)((op.nz + kTile - 1) / kTile));
  if (p_t)
    k_retile<false, true><<<g, 256, 0, s>>>(op, st, src_t, p_t, dst_k, nullptr, nullptr);
  else
    k_retile<false, false><<<g, 256, 0, s>>>(op, st, src_t, nullptr, dst_k, nullptr, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_precond_tiled(const Op& op, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s) {
  if (op.varying && op.recompute)
    k_precond_tiled_rc<true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  else if (op.varying)
    k_precond_tiled<true, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  else
    k_precond_tiled<false, true><<<grid, kTmThreads, 0, s>>>(op, st, r, q, z, partials, hist);
  return cudaGetLastError();
}

cudaError_t launch_spmv_tiled(const Op& op, DevState* st, const double* z, double* u, double* p,
                              double* q, double* partials, int grid, cudaStream_t s) {
  const int seglen = tiled_spmv_seglen(op, grid);
  if (op.varying && op.recompute)
    k_spmv_tiled<true, true><<<grid, 256, 0, s>>>(op, st, z, u, p, q, partials, seglen);
  else if (op.varying)
    k_spmv_tiled<true, false><<<grid, 256, 0, s>>>(op, st, z, u, p, q, partials, seglen);
  else
    k_spmv_tiled<false, false><<<grid, 256, 0, s>>>(op, st, z, u, p, q, partials, seglen);
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
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_spmv_tiled<true, false>, 256, 0);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_spmv_tiled<false, false>, 256, 0);
  long long g = (long long)std::max(1, b) * num_sms;
  // enough blocks for one unit per warp at the shortest segments
  const long long units = op.ntiles * std::max(1, op.nz / 4);
  const long long work = (units + 7) / 8;  // 8 warps per block
  if (g > work) g = work;
  return (int)(g < 1 ? 1 : g);
}

int grid_persistent(const Op& op, int num_sms) {
  int dev = 0, coop = 0, a = 0, b = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_pcg_persistent<true>, kPsThreads, 0) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_pcg_persistent<false>, kPsThreads, 0) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const int per_sm = std::min(a, b);
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
  const void* fn = op.varying ? reinterpret_cast<const void*>(k_pcg_persistent<true>)
                              : reinterpret_cast<const void*>(k_pcg_persistent<false>);
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kPsThreads), args, 0, s);
}

}  // namespace pcg
