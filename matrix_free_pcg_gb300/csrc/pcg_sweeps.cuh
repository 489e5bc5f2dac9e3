// Per-tile and per-unit bodies of the two row-tiled sweeps, shared by the
// sweep kernels (pcg_tiled.cu) and the persistent solve loop
// (pcg_persistent.cu); the row-tiled layout, cell (column c, level k) at
// (c/32*nz + k)*32 + c%32.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 6.1, eq. (22) (layout), Appendix A Algorithms 2 and 3 (sweeps).
#pragma once

#include <algorithm>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"

namespace pcg {
namespace {

// Preconditioner sweep: threads per block and levels per register chunk, of
// the forward pass (4 operands per level) and of the backward pass with
// per-cell factors (2 per level, one dependent fma: it needs twice the lead
// to cover an L2 round trip, in the registers the forward pass frees).
constexpr int kTmThreads = kTmWarpsPerBlock * 32;
constexpr int kTmChunk = 8;
constexpr int kTmChunkB = 16;
// The persistent loop's chunks (COHERENT): half as long, so that the whole
// loop fits 128 registers and runs 16 warps per SM.  Its grids have at most
// a few tiles per warp and live in L2, and its stencil phase needs the warps.
constexpr int kTmChunkP = 4;
constexpr int kTmChunkPB = 8;

__device__ __forceinline__ long long tiled_base(long long col, int nz) {
  return (col >> 5) * (long long)nz * kTile + (col & 31);
}

// One tile of the preconditioner sweep (see k_precond_tiled), for the lane's
// column: accumulates r*.r* and <r*, z> into accR, accK (FUSED).  COHERENT:
// q was written by other blocks of the same launch (the persistent loop), so
// it is read from L2, past the SM's non-coherent L1.  SCALE: z is stored as
// zscale * M^{-1} r (the damped line relaxation of the multigrid smoother),
// and <r*, z> is not accumulated (the smoother's caller reduces its own).
// FIRST (FUSED): the first sweep of a solve, where alpha = 0 and q was never
// written: r* = r, so q is not read and r not written back (fma(-0, q, r)
// with q = 0 is r, bit for bit).
template <bool VARY, bool FUSED, bool COHERENT = false, bool SCALE = false, bool FIRST = false>
__device__ __forceinline__ void precond_tile(const Op& op, long long t, int lane,
                                             double* __restrict__ r, const double* __restrict__ q,
                                             double* __restrict__ z, double nalpha, uint64_t keep,
                                             uint64_t stream, double& accR, double& accK,
                                             double zscale = 1.0) {
  const int nz = op.nz;
  const int fs = VARY ? kTile : 1;  // factor stride between levels
  if (t * kTile + lane >= op.ncols) return;
  const long long base = t * nz * kTile + lane;
  double* __restrict__ rt = r + base;
  const double* __restrict__ qt = FUSED ? q + base : nullptr;
  double* __restrict__ zt = z + base;
  const double* __restrict__ fi = VARY ? op.tinvd + base : op.lev + LV_INVD * nz;
  const double* __restrict__ fn = VARY ? op.tnphi + base : op.lev + LV_NPHI * nz;
  // ---- forward: level k uses nphi_{k-1} (0 at k = 0) and 1/D_k.  Only the w
  // scratch is marked to stay in L2 (evict-last) for the backward pass; the
  // factors' first read streams like the rest, though the backward pass reads
  // nphi again.  Kept as well, they crowded w out of L2: on 512x512x128 with
  // an a_h field ncu measured 55.2 B per cell and 0.385 ms per sweep, against
  // 53.9 B and 0.377 ms with nphi streamed.
  constexpr int CF = COHERENT ? kTmChunkP : kTmChunk;
  double cr[CF], cq[CF], ci[CF], cn[CF];
#pragma unroll
  for (int j = 0; j < CF; ++j) {
    const bool in = j < nz;
    cr[j] = in ? ld_hint(rt + j * kTile, stream) : 0.0;
    cq[j] = (FUSED && !FIRST && in)
                ? (COHERENT ? __ldcg(qt + j * kTile) : ld_hint(qt + j * kTile, stream))
                : 0.0;
    ci[j] = in ? (VARY ? ld_hint(fi + j * fs, stream) : __ldg(fi + j)) : 0.0;
    cn[j] = in ? (VARY ? ld_hint(fn + j * fs, stream) : __ldg(fn + j)) : 0.0;
  }
  double y = 0.0, nprev = 0.0, w = 0.0;
#pragma unroll 1
  for (int k0 = 0; k0 < nz; k0 += CF) {
    double nr[CF], nq[CF], ni[CF], nn[CF];
#pragma unroll
    for (int j = 0; j < CF; ++j) {
      const int k = k0 + CF + j;
      const bool in = k < nz;
      nr[j] = in ? ld_hint(rt + k * kTile, stream) : 0.0;
      nq[j] = (FUSED && !FIRST && in)
                  ? (COHERENT ? __ldcg(qt + k * kTile) : ld_hint(qt + k * kTile, stream))
                  : 0.0;
      ni[j] = in ? (VARY ? ld_hint(fi + k * fs, stream) : __ldg(fi + k)) : 0.0;
      nn[j] = in ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < CF; ++j) {
      const int k = k0 + j;
      if (k < nz) {
        double rk = cr[j];
        if (FUSED) {
          if (!FIRST) rk = fma(nalpha, cq[j], rk);
          accR = fma(rk, rk, accR);
          if (!FIRST) st_hint(rt + k * kTile, rk, stream);
        }
        y = fma(nprev, y, rk);
        w = y * ci[j];
        if (FUSED && !SCALE) accK = fma(y, w, accK);
        st_hint(zt + k * kTile, w, keep);
        nprev = cn[j];
      }
    }
#pragma unroll
    for (int j = 0; j < CF; ++j) {
      cr[j] = nr[j];
      cq[j] = nq[j];
      ci[j] = ni[j];
      cn[j] = nn[j];
    }
  }
  // ---- backward: z_{nz-1} = w_{nz-1} (in place); level k uses nphi_k.  With a
  // constant a_h the factors come from the per-level table and the longer
  // chunk costs registers (218 against 167): 8 levels there.
  constexpr int CB = COHERENT ? (VARY ? kTmChunkPB : kTmChunkP) : (VARY ? kTmChunkB : kTmChunk);
  // Chunk b holds levels kb, kb-1, ..., kb-CB+1 with kb = nz-2-b*CB.
  double zz = w;
  if (SCALE) st_hint(zt + (long long)(nz - 1) * kTile, w * zscale, stream);
  double bw[CB], bn[CB];
#pragma unroll
  for (int j = 0; j < CB; ++j) {
    const int k = nz - 2 - j;
    bw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
    bn[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
  }
#pragma unroll 1
  for (int kb = nz - 2; kb >= 0; kb -= CB) {
    double nw[CB], nb[CB];
#pragma unroll
    for (int j = 0; j < CB; ++j) {
      const int k = kb - CB - j;
      nw[j] = (k >= 0) ? ld_hint(zt + k * kTile, stream) : 0.0;
      nb[j] = (k >= 0) ? (VARY ? ld_hint(fn + k * fs, stream) : __ldg(fn + k)) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < CB; ++j) {
      const int k = kb - j;
      if (k >= 0) {
        zz = fma(bn[j], zz, bw[j]);
        st_hint(zt + k * kTile, SCALE ? zz * zscale : zz, stream);
      }
    }
#pragma unroll
    for (int j = 0; j < CB; ++j) {
      bw[j] = nw[j];
      bn[j] = nb[j];
    }
  }
}

// One unit (a segment of seglen levels of one tile) of the stencil sweep (see
// k_spmv_tiled) for the lane's column; accumulates <p, q> into sig.
//
// RESID: A z is formed as r + (A - M) z.  The preconditioner sweep has just
// solved M z = r, and M (eq. (19)) holds the whole diagonal of A and its
// vertical couplings, so A z - r is the horizontal neighbour sum alone:
// 4 fp64 operations per cell instead of 7, with r read in place of the
// diagonal.  Exact in real arithmetic; in floating point q differs from the
// explicit stencil by the column solve's backward error, of the same order
// (eps |A| |z|) as the stencil's own rounding.
//
// COHERENT: z and r were written by other blocks of the same launch (the
// persistent loop), so they are read from L2, past the SM's non-coherent L1.
//
// FIRST: the first sweep of a solve, where alpha = beta = 0 and p = q = 0 were
// never written: u keeps x0 (not read, not written), p = z and q = A z
// start from r (RESID) or the diagonal term alone, so neither u, p nor q is
// read -- 3 fp64 operations and 32 bytes per cell fewer.  The values are
// those of the general sweep with those zeros (fma(0, 0, v) = v), up to the
// sign of an exact zero.
template <bool VARY, bool RECOMP, bool RESID, bool COHERENT = false, bool FIRST = false>
__device__ __forceinline__ void spmv_unit(const Op& op, long long unit, int lane,
                                          const double* __restrict__ z,
                                          const double* __restrict__ r, double* __restrict__ u,
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
  const double sf = (RECOMP && !RESID) ? aE + aW + aN + aS : 0.0;
  auto ldz = [&](long long o) { return COHERENT ? __ldcg(z + o) : z[o]; };
  // the column window z_{k-1}, z_k, z_{k+1} (the explicit stencil only)
  double zd = (!RESID && k0 > 0) ? ldz(base + (long long)(k0 - 1) * kTile) : 0.0;
  double zc = RESID ? 0.0 : ldz(base + (long long)k0 * kTile);
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    const long long o = base + (long long)k * kTile;
    const long long ko = (long long)k * kTile;
    const double zu = (!RESID && k + 1 < nz) ? ldz(o + kTile) : 0.0;
    if (RESID) zc = ldz(o);
    const double zE = ldz(bE + ko), zW = ldz(bW + ko), zN = ldz(bN + ko), zS = ldz(bS + ko);
    double uc = FIRST ? 0.0 : __ldcs(u + o);
    double pc = FIRST ? 0.0 : __ldcs(p + o);
    const double qc = FIRST ? 0.0 : __ldcs(q + o);
    if (!FIRST) uc = fma(alpha, pc, uc);
    pc = FIRST ? zc : fma(beta, pc, zc);
    double a;
    if (VARY) {
      // per-cell horizontal weights -h_k a_f (west and south: the
      // neighbours' east and north weights), rebuilt with the set-up's
      // rounding under RECOMP
      double d = 0.0, cE, cW, cN, cS;
      if (RECOMP) {
        const double hw = __ldg(lev + LV_HW * nz + k);
        if (!RESID)
          d = __dadd_rn(__ldg(lev + LV_DIAG * nz + k), __dmul_rn(__ldg(lev + LV_H * nz + k), sf));
        cE = __dmul_rn(hw, aE);
        cW = __dmul_rn(hw, aW);
        cN = __dmul_rn(hw, aN);
        cS = __dmul_rn(hw, aS);
      } else {
        if (!RESID) d = __ldcs(op.cdiag_t + o);
        cE = __ldg(op.cwE_t + o);
        cW = __ldg(op.cwE_t + bW + ko);
        cN = __ldg(op.cwN_t + o);
        cS = __ldg(op.cwN_t + bS + ko);
      }
      if (RESID) {
        const double rc = COHERENT ? __ldcg(r + o) : __ldcs(r + o);
        a = FIRST ? rc : fma(beta, qc, rc);
      } else {
        a = FIRST ? d * zc : fma(d, zc, beta * qc);
        a = fma(__ldg(lev + LV_UP * nz + k), zu, a);
        a = fma(__ldg(lev + LV_DN * nz + k), zd, a);
      }
      a = fma(cE, zE, a);
      a = fma(cW, zW, a);
      a = fma(cN, zN, a);
      a = fma(cS, zS, a);
    } else {
      const double hs = (zE + zW) + (zN + zS);
      if (RESID) {
        const double rc = COHERENT ? __ldcg(r + o) : __ldcs(r + o);
        a = FIRST ? rc : fma(beta, qc, rc);
      } else {
        a = FIRST ? __ldg(lev + LV_DIAG * nz + k) * zc
                  : fma(__ldg(lev + LV_DIAG * nz + k), zc, beta * qc);
        a = fma(__ldg(lev + LV_UP * nz + k), zu, a);
        a = fma(__ldg(lev + LV_DN * nz + k), zd, a);
      }
      a = fma(__ldg(lev + LV_HW * nz + k), hs, a);
    }
    sig = fma(pc, a, sig);
    if (!FIRST) __stcs(u + o, uc);
    __stcs(p + o, pc);
    __stcs(q + o, a);
    if (!RESID) {
      zd = zc;
      zc = zu;
    }
  }
}

// Levels per work unit of the tiled stencil sweep: whole columns when there
// are at least 8 tiles per resident warp, else segments short enough to give
// every warp about 8 units (at least 4 levels each).
inline int tiled_spmv_seglen(const Op& op, int grid) {
  const long long warps = (long long)grid * 8;
  const long long want = 8 * warps;
  if (op.ntiles >= want || op.nz <= 4) return op.nz;
  long long nseg = (want + op.ntiles - 1) / op.ntiles;
  nseg = std::min<long long>(nseg, op.nz / 4);
  return (int)((op.nz + nseg - 1) / nseg);
}

}  // namespace
}  // namespace pcg
