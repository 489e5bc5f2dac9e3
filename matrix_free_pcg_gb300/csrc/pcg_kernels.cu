// Device kernels of the matrix-free PCG solver (fp64, sm_103a) for the
// column-contiguous layout, plus the stencil kernels every layout uses (the
// standalone operator and the initial residual) and the deferred update.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs".
//   - stencil: section 4.2, eq. (18), recomputed from per-level tables
//     (eq. (17)) and per-column face values;
//   - column preconditioner: section 4.1 and eq. (19), Thomas algorithm;
//   - fused sweeps: section 4.3, Algorithm 1, with the two kernels of
//     Appendix A (Algorithm 2: SpMV sweep, Algorithm 3: preconditioner sweep).
//
// Design for GB300.  The fp64 pipe of this part retires 2 lane operations per
// SM per clock at most, so at the 88-112 bytes per cell and iteration that
// these sweeps move, the iteration is bound by fp64 arithmetic, not by HBM.
// The kernels therefore spend integer and load/store instructions freely and
// keep the fp64 instruction count at the minimum of the formulation: 6 per
// cell in the preconditioner sweep, 11 (constant a_h) or 12 (a_h per column:
// face values per column) in the stencil sweep.  Both sweeps are persistent
// grids (a few blocks per SM), so the per-thread partial sums are folded into
// the grid reduction only once per launch.
//
// Vectors use the column-contiguous layout: cell (i,j,k) at ((j*nx)+i)*nz+k.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "pcg_internal.h"
#include "pcg_device.cuh"

namespace pcg {
namespace {

// acc + (A z) at the two cells l, l+1 of one column (k even, k+1 < nz),
// eq. (18).  zc = (z[l], z[l+1]).  The vertical neighbours outside the column
// enter with a zero coefficient (Neumann lid and floor).
template <bool VARY>
__device__ __forceinline__ double2 stencil2(const Op& op, const double* __restrict__ z,
                                            long long l, long long col, int k, double2 acc,
                                            double2 zc) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const Nbr nb = neighbours(op, col);
  const double zd = (k > 0) ? z[l - 1] : 0.0;
  const double zu = (k + 2 < nz) ? z[l + 2] : 0.0;
  const double2 zE = ld2(z + nb.e * nz + k);
  const double2 zW = ld2(z + nb.w * nz + k);
  const double2 zN = ld2(z + nb.n * nz + k);
  const double2 zS = ld2(z + nb.s * nz + k);
  double h0, h1, d0, d1;
  if (VARY) {
    const double aE = __ldg(op.faceE + col), aW = __ldg(op.faceE + nb.w);
    const double aN = __ldg(op.faceN + col), aS = __ldg(op.faceN + nb.s);
    h0 = aE * zE.x;
    h0 = fma(aW, zW.x, h0);
    h0 = fma(aN, zN.x, h0);
    h0 = fma(aS, zS.x, h0);
    h1 = aE * zE.y;
    h1 = fma(aW, zW.y, h1);
    h1 = fma(aN, zN.y, h1);
    h1 = fma(aS, zS.y, h1);
    const double2 dg = ldg2(op.cdiag + l);
    d0 = dg.x;
    d1 = dg.y;
  } else {
    h0 = (zE.x + zW.x) + (zN.x + zS.x);
    h1 = (zE.y + zW.y) + (zN.y + zS.y);
    d0 = __ldg(lev + LV_DIAG * nz + k);
    d1 = __ldg(lev + LV_DIAG * nz + k + 1);
  }
  double a0 = fma(d0, zc.x, acc.x);
  a0 = fma(__ldg(lev + LV_UP * nz + k), zc.y, a0);
  a0 = fma(__ldg(lev + LV_DN * nz + k), zd, a0);
  a0 = fma(__ldg(lev + LV_HW * nz + k), h0, a0);
  double a1 = fma(d1, zc.y, acc.y);
  a1 = fma(__ldg(lev + LV_UP * nz + k + 1), zu, a1);
  a1 = fma(__ldg(lev + LV_DN * nz + k + 1), zc.x, a1);
  a1 = fma(__ldg(lev + LV_HW * nz + k + 1), h1, a1);
  return make_double2(a0, a1);
}

// acc + (A z) at one cell l (any nz, any alignment).
template <bool VARY>
__device__ __forceinline__ double stencil1(const Op& op, const double* __restrict__ z,
                                           long long l, long long col, int k, double acc,
                                           double zc) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const Nbr nb = neighbours(op, col);
  const double zd = (k > 0) ? z[l - 1] : 0.0;
  const double zu = (k + 1 < nz) ? z[l + 1] : 0.0;
  const double zE = z[nb.e * nz + k], zW = z[nb.w * nz + k];
  const double zN = z[nb.n * nz + k], zS = z[nb.s * nz + k];
  double hs, d;
  if (VARY) {
    hs = __ldg(op.faceE + col) * zE;
    hs = fma(__ldg(op.faceE + nb.w), zW, hs);
    hs = fma(__ldg(op.faceN + col), zN, hs);
    hs = fma(__ldg(op.faceN + nb.s), zS, hs);
    d = __ldg(op.cdiag + l);
  } else {
    hs = (zE + zW) + (zN + zS);
    d = __ldg(lev + LV_DIAG * nz + k);
  }
  double a = fma(d, zc, acc);
  a = fma(__ldg(lev + LV_UP * nz + k), zu, a);
  a = fma(__ldg(lev + LV_DN * nz + k), zd, a);
  return fma(__ldg(lev + LV_HW * nz + k), hs, a);
}

// ------------------------------------------------- preconditioner sweep (K_M)

// Shared-memory index of level k of a staged column: XOR swizzle of the low
// four bits with the column's position in the tile, so that 16 threads that
// read the same level of 16 different columns hit 16 distinct 8-byte bank
// pairs (column stride pz is a multiple of 16 doubles).
struct SwzIdx {
  int sw;
  __device__ __forceinline__ int operator()(int k) const { return k ^ sw; }
};
struct LinIdx {
  __device__ __forceinline__ int operator()(int k) const { return k; }
};

// Copy cnt = nc*nz consecutive doubles (nc whole columns) from global memory
// into the swizzled tile, cooperatively by the 32 lanes of the warp (used for
// odd nz or 8-byte aligned vectors, where the bulk-copy engine cannot be).
__device__ __forceinline__ void tile_load(const double* __restrict__ g, double* s, int cnt,
                                          int nz, int pz, int lane) {
  int e = lane, c = e / nz, k = e - c * nz;
  for (; e < cnt; e += 32) {
    s[c * pz + (k ^ (c & 15))] = g[e];
    k += 32;
    while (k >= nz) {
      k -= nz;
      ++c;
    }
  }
}

__device__ __forceinline__ void tile_store(const double* s, double* __restrict__ g, int cnt,
                                           int nz, int pz, int lane) {
  int e = lane, c = e / nz, k = e - c * nz;
  for (; e < cnt; e += 32) {
    g[e] = s[c * pz + (k ^ (c & 15))];
    k += 32;
    while (k >= nz) {
      k -= nz;
      ++c;
    }
  }
}

// One column of Algorithm 3 (FUSED) or of the plain solve M z = r.
//   rp: r on entry; with FUSED r* = r - alpha q on exit.
//   qp: q (FUSED only).  wp: receives z (may alias qp: q_k is read before
//   w_k overwrites it).
// Forward: y_k = r*_k + (T_{k-1/2}/D_{k-1}) y_{k-1},  w_k = y_k / D_k;
// backward: z_k = w_k + (T_{k+1/2}/D_k) z_{k+1}.  fp64 operations per level:
// 4 forward (r*, ||r||^2, y, w), 2 backward (z, <r,z>).
//
// The two Thomas factors of every level are loaded kPre levels ahead of their
// use into registers, so their global-memory latency overlaps the serial
// recurrence instead of sitting inside it.
constexpr int kPre = 16;

template <bool VARY, bool FUSED, typename IDX>
__device__ __forceinline__ void column_solve(const Op& op, long long tile, int lane, IDX idx,
                                             double* rp, const double* qp, double* wp,
                                             double nalpha, double& accR, double& accK) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const double* __restrict__ fn = VARY ? op.tnphi + tile * nz * kTile + lane : lev + LV_NPHI * nz;
  const double* __restrict__ fi = VARY ? op.tinvd + tile * nz * kTile + lane : lev + LV_INVD * nz;
  const int fs = VARY ? kTile : 1;
  // ---- forward elimination; level k uses nphi_{k-1} (0 at k = 0) and invd_k
  double cn[kPre], ci[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    cn[j] = (j >= 1 && j - 1 < nz) ? __ldg(fn + (j - 1) * fs) : 0.0;
    ci[j] = (j < nz) ? __ldg(fi + j * fs) : 0.0;
  }
  double y = 0.0;
  for (int kc = 0; kc < nz; kc += kPre) {
    double nn[kPre], ni[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = kc + kPre + j;
      nn[j] = (k - 1 < nz) ? __ldg(fn + (k - 1) * fs) : 0.0;
      ni[j] = (k < nz) ? __ldg(fi + k * fs) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = kc + j;
      if (k < nz) {
        const int o = idx(k);
        double rk = rp[o];
        if (FUSED) {
          rk = fma(nalpha, qp[o], rk);
          accR = fma(rk, rk, accR);
          rp[o] = rk;
        }
        y = fma(cn[j], y, rk);
        wp[o] = y * ci[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      cn[j] = nn[j];
      ci[j] = ni[j];
    }
  }
  // ---- back substitution; level k uses nphi_k
  int o = idx(nz - 1);
  double zz = wp[o];
  if (FUSED) accK = fma(zz, rp[o], accK);
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int k = nz - 2 - j;
    cn[j] = (k >= 0) ? __ldg(fn + k * fs) : 0.0;
  }
  for (int kb = nz - 2; kb >= 0; kb -= kPre) {
    double nn[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = kb - kPre - j;
      nn[j] = (k >= 0) ? __ldg(fn + k * fs) : 0.0;
    }
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int k = kb - j;
      if (k >= 0) {
        o = idx(k);
        zz = fma(cn[j], zz, wp[o]);
        wp[o] = zz;
        if (FUSED) accK = fma(zz, rp[o], accK);
      }
    }
#pragma unroll
    for (int j = 0; j < kPre; ++j) cn[j] = nn[j];
  }
}

template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTile) k_precond_staged(Op op, DevState* st,
                                                          double* __restrict__ r,
                                                          const double* __restrict__ q,
                                                          double* __restrict__ z,
                                                          double* __restrict__ partials,
                                                          double* __restrict__ hist) {
  extern __shared__ double smem[];
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x;
  const int nz = op.nz, pz = op.pz;
  double* sr = smem;
  double* sq = smem + kTile * pz;
  const double nalpha = FUSED ? -st->alpha : 0.0;
  double accR = 0.0, accK = 0.0;
  const SwzIdx idx{lane & 15};
  for (long long t = blockIdx.x; t < op.ntiles; t += gridDim.x) {
    const long long col0 = t * kTile;
    const int nc = (int)min((long long)kTile, op.ncols - col0);
    const long long base = col0 * nz;
    const int cnt = nc * nz;
    tile_load(r + base, sr, cnt, nz, pz, lane);
    if (FUSED) tile_load(q + base, sq, cnt, nz, pz, lane);
    __syncwarp();
    if (lane < nc)
      column_solve<VARY, FUSED>(op, t, lane, idx, sr + lane * pz, sq + lane * pz,
                                sq + lane * pz, nalpha, accR, accK);
    __syncwarp();
    if (FUSED) tile_store(sr, r + base, cnt, nz, pz, lane);
    tile_store(sq, z + base, cnt, nz, pz, lane);
    __syncwarp();
  }
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTile>(accR, accK, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

// Streaming variant (nz even, 16-byte aligned vectors), the main path.
//
// Only w, the result of the forward sweep that the backward sweep consumes in
// reverse, stays in shared memory for a whole column (tile W, 32 columns at
// an even stride pt = 2 (mod 4) doubles, at most 2-way bank conflicts).  r
// and q stream through rings of kStages slots of kChunk levels, filled two
// chunks ahead by 16-byte asynchronous copies (cp.async) in a transposed
// lane mapping: four lanes cover the 64 bytes of one column's chunk, so one
// instruction moves 8 columns x 64 contiguous bytes.  r* = r - alpha q is
// written back into its ring slot and then to global memory, and z from W at
// the end of the column, with the same coalesced mapping.  At nz = 128 this
// is 48.7 KB of shared memory per warp: four warps per SM, the number the
// SM's fp64 unit needs to run at full rate (a single warp issues one fp64
// instruction about every 68 clocks).  The launch sizes its shared-memory
// request so that the warps per SM are a multiple of four.
//
// <r,z> is accumulated in the forward sweep as sum_k y_k w_k: with
// y = L^{-1} r* and w = D^{-1} y this is r*^T L^{-T} D^{-1} L^{-1} r* =
// <r*, M^{-1} r*>, the same number Algorithm 3 sums in its backward loop.
constexpr int kChunk = 16;
constexpr int kStages = 2;
constexpr int kCS = kChunk + 2;  // ring row (doubles): 144 B, 16-byte aligned, no 16-byte conflicts
// Dynamic shared memory the streaming kernels may request: the per-block
// opt-in limit minus their static shared memory (set in prepare_kernels).
static int g_max_stream_smem = 0;

template <bool FUSED>
__host__ __device__ inline size_t stream_smem_bytes(int pt) {
  return sizeof(double) * ((size_t)kTile * pt + (FUSED ? 2 : 1) * (size_t)kStages * kTile * kCS);
}

// FULL: nz is a multiple of kChunk (no partial chunk, no guards).
template <bool VARY, bool FUSED, bool FULL>
__global__ void __launch_bounds__(kTile) k_precond_stream(Op op, DevState* st,
                                                          double* __restrict__ r,
                                                          const double* __restrict__ q,
                                                          double* __restrict__ z,
                                                          double* __restrict__ partials,
                                                          double* __restrict__ hist) {
  extern __shared__ __align__(16) double smem[];
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x;
  const int nz = op.nz, pt = op.pt;
  const int nch = (nz + kChunk - 1) / kChunk;
  double* W = smem;
  double* Rg = W + kTile * pt;
  double* Qg = Rg + kStages * kTile * kCS;
  const double nalpha = FUSED ? -st->alpha : 0.0;
  const double* __restrict__ lev = op.lev;
  // Transposed roles for the coalesced copies: eight lanes cover the 128
  // bytes of one column's chunk, so one instruction moves 4 columns x 128
  // contiguous bytes.  Lane handles columns cq + 4i, 16-byte piece pp.
  const int cq = lane >> 3, pp = 2 * (lane & 7);
  double accR0 = 0.0, accR1 = 0.0, accK0 = 0.0, accK1 = 0.0;
  // Static tile assignment (block b takes tiles b, b+G, ...): the per-block
  // partial sums, and with them the reductions, are the same on every run.
  const long long G = gridDim.x;
  long long p_tile = blockIdx.x;
  int p_m = 0, p_sl = 0;
  // Producer: the copies of the next chunk in (tile, chunk) order, one
  // commit group per chunk (possibly empty past the last tile).
  auto issue = [&]() {
    if (p_tile < op.ntiles) {
      const long long col0 = p_tile * kTile;
      const int nc = (int)min((long long)kTile, op.ncols - col0);
      const int k0 = p_m * kChunk;
      const int clen = FULL ? kChunk : min(kChunk, nz - k0);
      if (FULL || pp < clen) {
        const double* rsrc = r + (col0 + cq) * nz + k0 + pp;
        const double* qsrc = FUSED ? q + (col0 + cq) * nz + k0 + pp : nullptr;
        double* rdst = Rg + (p_sl * kTile + cq) * kCS + pp;
        double* qdst = Qg + (p_sl * kTile + cq) * kCS + pp;
#pragma unroll
        for (int i = 0; i < kTile / 4; ++i) {
          if (cq + 4 * i < nc) {
            cp_async16(rdst + 4 * i * kCS, rsrc + (long long)4 * i * nz);
            if (FUSED) cp_async16(qdst + 4 * i * kCS, qsrc + (long long)4 * i * nz);
          }
        }
      }
    }
    cp_async_commit();
    if (++p_m == nch) {
      p_m = 0;
      p_tile += G;
    }
    p_sl ^= 1;
  };
  issue();  // prologue: chunk 0
  int c_sl = 0;
  for (long long t = blockIdx.x; t < op.ntiles; t += G) {
    const long long col0 = t * kTile;
    const int nc = (int)min((long long)kTile, op.ncols - col0);
    double* wcol = W + lane * pt;
    const double* fi = VARY ? op.tinvd + t * nz * kTile + lane : lev + LV_INVD * nz;
    const double* fn = VARY ? op.tnphi + t * nz * kTile + lane : lev + LV_NPHI * nz;
    const int fs = VARY ? kTile : 1;
    double y = 0.0, nprev = 0.0;
    double cfi[kChunk], cfn[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      cfi[j] = (FULL || j < nz) ? __ldg(fi + j * fs) : 0.0;
      cfn[j] = (FULL || j < nz) ? __ldg(fn + j * fs) : 0.0;
    }
    // ---- forward sweep, chunk by chunk
#pragma unroll 1
    for (int m = 0; m < nch; ++m) {
      const int k0 = m * kChunk;
      const int clen = FULL ? kChunk : min(kChunk, nz - k0);
      issue();                 // chunk seq+1 into the slot of chunk seq-1
      double nfi[kChunk], nfn[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        const int k = k0 + kChunk + j;
        nfi[j] = (k < nz) ? __ldg(fi + k * fs) : 0.0;
        nfn[j] = (k < nz) ? __ldg(fn + k * fs) : 0.0;
      }
      cp_async_wait<1>();      // this lane's copies of chunk seq have landed
      __syncwarp();            // ... and everyone else's
      if (lane < nc) {
        double* rs = Rg + (c_sl * kTile + lane) * kCS;
        const double* qs = Qg + (c_sl * kTile + lane) * kCS;
#pragma unroll
        for (int j = 0; j < kChunk; j += 2) {
          if (FULL || j < clen) {
            const double2 rv = lds2(rs + j);
            double r0 = rv.x, r1 = rv.y;
            if (FUSED) {
              const double2 qv = lds2(qs + j);
              r0 = fma(nalpha, qv.x, r0);
              r1 = fma(nalpha, qv.y, r1);
              accR0 = fma(r0, r0, accR0);
              accR1 = fma(r1, r1, accR1);
              sts2(rs + j, r0, r1);
            }
            y = fma(nprev, y, r0);
            const double w0 = y * cfi[j];
            if (FUSED) accK0 = fma(y, w0, accK0);
            y = fma(cfn[j], y, r1);
            const double w1 = y * cfi[j + 1];
            if (FUSED) accK1 = fma(y, w1, accK1);
            nprev = cfn[j + 1];
            sts2(wcol + k0 + j, w0, w1);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        cfi[j] = nfi[j];
        cfn[j] = nfn[j];
      }
      __syncwarp();
      if (FUSED && (FULL || pp < clen)) {  // r* of this chunk back to global memory
        double* rdst = r + (col0 + cq) * nz + k0 + pp;
        const double* rsrc = Rg + (c_sl * kTile + cq) * kCS + pp;
#pragma unroll
        for (int i = 0; i < kTile / 4; ++i)
          if (cq + 4 * i < nc) st2(rdst + (long long)4 * i * nz, lds2(rsrc + 4 * i * kCS));
      }
      __syncwarp();  // the slot is refilled by the next issue()
      c_sl ^= 1;
    }
    // ---- backward sweep over W (nz is even here).  Level nz-1 is final;
    // level nz-2 alone; then pairs (kh-1, kh), kh = nz-3, nz-5, ..., 1, each
    // read and written as one 16-byte pair.  Factor s of the pair sequence
    // belongs to level nz-3-s and is loaded kPre levels ahead.
    if (lane < nc) {
      double zz = wcol[nz - 1];
      if (nz >= 2) {
        zz = fma(__ldg(fn + (nz - 2) * fs), zz, wcol[nz - 2]);
        wcol[nz - 2] = zz;
      }
      double cn[kPre];
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const int k = nz - 3 - j;
        cn[j] = (k >= 0) ? __ldg(fn + k * fs) : 0.0;
      }
#pragma unroll 1
      for (int sb = 0; sb < nz - 2; sb += kPre) {
        double nn[kPre];
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
          const int k = nz - 3 - (sb + kPre + j);
          nn[j] = (k >= 0) ? __ldg(fn + k * fs) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < kPre; j += 2) {
          const int kh = nz - 3 - (sb + j);  // odd
          if (kh >= 1) {
            const double2 wv = lds2(wcol + kh - 1);
            const double zh = fma(cn[j], zz, wv.y);
            zz = fma(cn[j + 1], zh, wv.x);
            sts2(wcol + kh - 1, zz, zh);
          }
        }
#pragma unroll
        for (int j = 0; j < kPre; ++j) cn[j] = nn[j];
      }
    }
    __syncwarp();
    // z of the whole tile to global memory, 4 columns x 128 bytes per store
    {
      double* zdst = z + (col0 + cq) * nz + pp;
      const double* wsrc = W + cq * pt + pp;
#pragma unroll
      for (int i = 0; i < kTile / 4; ++i) {
        if (cq + 4 * i < nc) {
          for (int k = 0; k < nz; k += kChunk)
            if (FULL || pp + k < nz)
              st2(zdst + (long long)4 * i * nz + k, lds2(wsrc + 4 * i * pt + k));
        }
      }
    }
    __syncwarp();  // W is rewritten by the next tile
  }
  cp_async_wait<0>();
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTile>(accR0 + accR1, accK0 + accK1, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

// Column-height-specialised variant of the streaming sweep (nz = 32, 64,
// 128: the heights of the workloads), the main path for those heights.
//
// It keeps the data flow of k_precond_stream for r, q and r*, with every
// level loop unrolled at compile time.  w, the forward result the backward
// sweep consumes in reverse, does not stay in shared memory: each block owns
// a private scratch region in global memory (32 x NZ doubles, level-major,
// so that one level of the 32 columns is one 256-byte line), written in the
// forward sweep and read back, still resident in L2, in the backward sweep.
// Shared memory then holds only the two r/q rings (18.4 KB), so eight warps
// -- two per SM sub-partition -- fit on an SM and hide each other's
// latencies; with one warp per sub-partition every dependent instruction
// waits out a full fp64 latency.  z leaves through the ring slot that is
// free during the backward sweep, transposed for coalesced stores.
template <int NZ, bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTile) k_precond_fixed(Op op, DevState* st,
                                                         double* __restrict__ r,
                                                         const double* __restrict__ q,
                                                         double* __restrict__ z,
                                                         double* __restrict__ partials,
                                                         double* __restrict__ hist) {
  constexpr int NCH = NZ / kChunk;
  constexpr int FS = VARY ? kTile : 1;  // factor stride between levels
  static_assert(NZ % (2 * kChunk) == 0, "an even number of whole chunks");
  extern __shared__ __align__(16) double smem[];
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x;
  double* Rg = smem;
  double* Qg = Rg + kStages * kTile * kCS;
  double* wsb = op.wscratch + (long long)blockIdx.x * NZ * kTile + lane;  // level k at wsb[k*32]
  const double nalpha = FUSED ? -st->alpha : 0.0;
  const int cq = lane >> 3, pp = 2 * (lane & 7);
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accR0 = 0.0, accR1 = 0.0, accK0 = 0.0, accK1 = 0.0;
  // factor loads: per-cell arrays stream through L2 (nphi is read twice);
  // the per-level table of a constant a_h stays in L1
  auto ldf = [&](const double* a, uint64_t pol) { return VARY ? ld_hint(a, pol) : __ldg(a); };
  const long long G = gridDim.x;
  // copies of chunk m of tile t into ring slot sl (whole warp), one group
  auto issue = [&](long long t, int m, int sl) {
    if (t < op.ntiles) {
      const long long col0 = t * kTile;
      const int nc = (int)min((long long)kTile, op.ncols - col0);
      const double* rsrc = r + (col0 + cq) * NZ + m * kChunk + pp;
      const double* qsrc = FUSED ? q + (col0 + cq) * NZ + m * kChunk + pp : nullptr;
      double* rdst = Rg + (sl * kTile + cq) * kCS + pp;
      double* qdst = Qg + (sl * kTile + cq) * kCS + pp;
#pragma unroll
      for (int i = 0; i < kTile / 4; ++i) {
        if (cq + 4 * i < nc) {
          cp_async16_hint(rdst + 4 * i * kCS, rsrc + 4 * i * NZ, stream);
          if (FUSED) cp_async16_hint(qdst + 4 * i * kCS, qsrc + 4 * i * NZ, stream);
        }
      }
    }
    cp_async_commit();
  };
  issue(blockIdx.x, 0, 0);
  for (long long t = blockIdx.x; t < op.ntiles; t += G) {
    const long long col0 = t * kTile;
    const int nc = (int)min((long long)kTile, op.ncols - col0);
    const double* __restrict__ fi =
        VARY ? op.tinvd + t * NZ * kTile + lane : op.lev + LV_INVD * NZ;
    const double* __restrict__ fn =
        VARY ? op.tnphi + t * NZ * kTile + lane : op.lev + LV_NPHI * NZ;
    double y = 0.0, nprev = 0.0;
    double ci[kChunk], cn[kChunk], ww[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      ci[j] = ldf(fi + j * FS, stream);
      cn[j] = ldf(fn + j * FS, keep);
    }
    // ---- forward sweep
#pragma unroll 1
    for (int m = 0; m < NCH; ++m) {
      const int sl = m & 1;
      if (m + 1 < NCH)
        issue(t, m + 1, (m + 1) & 1);
      else
        issue(t + G, 0, 0);
      double ni[kChunk], nn[kChunk];
      if (m + 1 < NCH) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          ni[j] = ldf(fi + ((m + 1) * kChunk + j) * FS, stream);
          nn[j] = ldf(fn + ((m + 1) * kChunk + j) * FS, keep);
        }
      }
      cp_async_wait<1>();
      __syncwarp();
      if (lane < nc) {
        double* rs = Rg + (sl * kTile + lane) * kCS;
        const double* qs = Qg + (sl * kTile + lane) * kCS;
#pragma unroll
        for (int j = 0; j < kChunk; j += 2) {
          const double2 rv = lds2(rs + j);
          double r0 = rv.x, r1 = rv.y;
          if (FUSED) {
            const double2 qv = lds2(qs + j);
            r0 = fma(nalpha, qv.x, r0);
            r1 = fma(nalpha, qv.y, r1);
            accR0 = fma(r0, r0, accR0);
            accR1 = fma(r1, r1, accR1);
            sts2(rs + j, r0, r1);
          }
          y = fma(nprev, y, r0);
          ww[j] = y * ci[j];
          if (FUSED) accK0 = fma(y, ww[j], accK0);
          y = fma(cn[j], y, r1);
          ww[j + 1] = y * ci[j + 1];
          if (FUSED) accK1 = fma(y, ww[j + 1], accK1);
          nprev = cn[j + 1];
        }
        if (m + 1 < NCH) {  // the last chunk's w stays in registers for the backward sweep
#pragma unroll
          for (int j = 0; j < kChunk; ++j) st_hint(wsb + (m * kChunk + j) * kTile, ww[j], keep);
        }
      }
      __syncwarp();
      if (FUSED) {
        double* rdst = r + (col0 + cq) * NZ + m * kChunk + pp;
        const double* rsrc = Rg + (sl * kTile + cq) * kCS + pp;
#pragma unroll
        for (int i = 0; i < kTile / 4; ++i)
          if (cq + 4 * i < nc) st2_hint(rdst + 4 * i * NZ, lds2(rsrc + 4 * i * kCS), stream);
      }
      __syncwarp();
      if (m + 1 < NCH) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          ci[j] = ni[j];
          cn[j] = nn[j];
        }
      }
    }
    // ---- backward sweep, chunk by chunk from the top; w of the top chunk is
    // in registers, the others come back from the scratch region.  Each
    // finished chunk of z is staged in ring slot 1 (free now: the producer's
    // next copy went to slot 0) and stored transposed.
    double* zs = Rg + (kTile + lane) * kCS;
    double bw[kChunk], bn[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      bw[j] = ww[j];
      bn[j] = ldf(fn + ((NCH - 1) * kChunk + j) * FS, stream);
    }
    double zz = 0.0;
#pragma unroll 1
    for (int c = NCH - 1; c >= 0; --c) {
      double nw[kChunk], nb[kChunk];
      if (c > 0 && lane < nc) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          nw[j] = ld_hint(wsb + ((c - 1) * kChunk + j) * kTile, stream);
          nb[j] = ldf(fn + ((c - 1) * kChunk + j) * FS, stream);
        }
      }
      if (lane < nc) {
#pragma unroll
        for (int j = kChunk - 1; j >= 1; j -= 2) {
          const int k = c * kChunk + j;
          const double zh = (k == NZ - 1) ? bw[j] : fma(bn[j], zz, bw[j]);
          zz = fma(bn[j - 1], zh, bw[j - 1]);
          sts2(zs + j - 1, zz, zh);
        }
      }
      __syncwarp();
      {
        double* zdst = z + (col0 + cq) * NZ + c * kChunk + pp;
        const double* zsrc = Rg + (kTile + cq) * kCS + pp;
#pragma unroll
        for (int i = 0; i < kTile / 4; ++i)
          if (cq + 4 * i < nc) st2_hint(zdst + 4 * i * NZ, lds2(zsrc + 4 * i * kCS), stream);
      }
      __syncwarp();
      if (c > 0) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          bw[j] = nw[j];
          bn[j] = nb[j];
        }
      }
    }
  }
  cp_async_wait<0>();
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTile>(accR0 + accR1, accK0 + accK1, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

template <bool FUSED>
__host__ __device__ inline size_t fixed_smem_bytes() {
  return sizeof(double) * (FUSED ? 2 : 1) * (size_t)kStages * kTile * kCS;
}

// Unstaged variant for columns too tall for the shared-memory tile: each
// thread walks its column in global memory (correct for any nz; the
// reduction and bookkeeping are those of the staged kernel).
template <bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTile) k_precond_direct(Op op, DevState* st,
                                                          double* __restrict__ r,
                                                          const double* __restrict__ q,
                                                          double* __restrict__ z,
                                                          double* __restrict__ partials,
                                                          double* __restrict__ hist) {
  if (FUSED && ld_done(st)) return;
  const int lane = threadIdx.x;
  const int nz = op.nz;
  const double nalpha = FUSED ? -st->alpha : 0.0;
  double accR = 0.0, accK = 0.0;
  for (long long t = blockIdx.x; t < op.ntiles; t += gridDim.x) {
    const long long col = t * kTile + lane;
    if (col < op.ncols)
      column_solve<VARY, FUSED>(op, t, lane, LinIdx{}, r + col * nz, FUSED ? q + col * nz : nullptr,
                                z + col * nz, nalpha, accR, accK);
  }
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTile>(accR, accK, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

// acc + ((A - M) z) at the two cells l, l+1 of one column: the horizontal
// neighbour terms alone (M, eq. (19), holds A's diagonal and vertical
// couplings).  acc = r + beta q turns it into A z + beta q for the z of
// M z = r (the residual form of the stencil sweep).
template <bool VARY>
__device__ __forceinline__ double2 horizontal2(const Op& op, const double* __restrict__ z,
                                               long long l, long long col, int k, double2 acc) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const Nbr nb = neighbours(op, col);
  const double2 zE = ld2(z + nb.e * nz + k);
  const double2 zW = ld2(z + nb.w * nz + k);
  const double2 zN = ld2(z + nb.n * nz + k);
  const double2 zS = ld2(z + nb.s * nz + k);
  double h0, h1;
  if (VARY) {
    const double aE = __ldg(op.faceE + col), aW = __ldg(op.faceE + nb.w);
    const double aN = __ldg(op.faceN + col), aS = __ldg(op.faceN + nb.s);
    h0 = aE * zE.x;
    h0 = fma(aW, zW.x, h0);
    h0 = fma(aN, zN.x, h0);
    h0 = fma(aS, zS.x, h0);
    h1 = aE * zE.y;
    h1 = fma(aW, zW.y, h1);
    h1 = fma(aN, zN.y, h1);
    h1 = fma(aS, zS.y, h1);
  } else {
    h0 = (zE.x + zW.x) + (zN.x + zS.x);
    h1 = (zE.y + zW.y) + (zN.y + zS.y);
  }
  return make_double2(fma(__ldg(lev + LV_HW * nz + k), h0, acc.x),
                      fma(__ldg(lev + LV_HW * nz + k + 1), h1, acc.y));
}

// acc + ((A - M) z) at one cell l.
template <bool VARY>
__device__ __forceinline__ double horizontal1(const Op& op, const double* __restrict__ z,
                                              long long l, long long col, int k, double acc) {
  const int nz = op.nz;
  const Nbr nb = neighbours(op, col);
  const double zE = z[nb.e * nz + k], zW = z[nb.w * nz + k];
  const double zN = z[nb.n * nz + k], zS = z[nb.s * nz + k];
  double hs;
  if (VARY) {
    hs = __ldg(op.faceE + col) * zE;
    hs = fma(__ldg(op.faceE + nb.w), zW, hs);
    hs = fma(__ldg(op.faceN + col), zN, hs);
    hs = fma(__ldg(op.faceN + nb.s), zS, hs);
  } else {
    hs = (zE + zW) + (zN + zS);
  }
  return fma(__ldg(op.lev + LV_HW * nz + k), hs, acc);
}

// ----------------------------------------------------- stencil sweeps (K_A)

// Algorithm 2: u += alpha p; p = z + beta p; q = A z + beta q; sigma = <p,q>;
// then alpha = kappa_old / sigma in the last block.  RESID: A z = r + (A - M) z
// for the z of M z = r from the preconditioner sweep (horizontal terms only).
template <bool VARY, bool VEC2, bool RESID>
__global__ void __launch_bounds__(kSpmvThreads) k_spmv_fused(Op op, DevState* st,
                                                             const double* __restrict__ z,
                                                             const double* __restrict__ r,
                                                             double* __restrict__ u,
                                                             double* __restrict__ p,
                                                             double* __restrict__ q,
                                                             double* __restrict__ partials) {
  if (ld_done(st)) return;
  const double alpha = st->alpha, beta = st->beta;
  const int nz = op.nz;
  double sig = 0.0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC2) {
    const long long np = op.n >> 1;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < np; g += stride) {
      const long long l = g << 1;
      const long long col = l / nz;
      const int k = (int)(l - col * nz);
      const double2 zc = ld2(z + l);
      double2 pc = ld2(p + l);
      const double2 qc = ld2(q + l);
      double2 uc = ld2(u + l);
      uc.x = fma(alpha, pc.x, uc.x);
      uc.y = fma(alpha, pc.y, uc.y);
      pc.x = fma(beta, pc.x, zc.x);
      pc.y = fma(beta, pc.y, zc.y);
      double2 qn;
      if (RESID) {
        const double2 rc = ld2(r + l);
        qn = horizontal2<VARY>(op, z, l, col, k,
                               make_double2(fma(beta, qc.x, rc.x), fma(beta, qc.y, rc.y)));
      } else {
        qn = stencil2<VARY>(op, z, l, col, k, make_double2(beta * qc.x, beta * qc.y), zc);
      }
      sig = fma(pc.x, qn.x, sig);
      sig = fma(pc.y, qn.y, sig);
      st2(u + l, uc);
      st2(p + l, pc);
      st2(q + l, qn);
    }
  } else {
    for (long long l = blockIdx.x * (long long)blockDim.x + threadIdx.x; l < op.n; l += stride) {
      const long long col = l / nz;
      const int k = (int)(l - col * nz);
      const double zc = z[l];
      const double pc = fma(beta, p[l], zc);
      u[l] = fma(alpha, p[l], u[l]);
      const double qn = RESID ? horizontal1<VARY>(op, z, l, col, k, fma(beta, q[l], r[l]))
                              : stencil1<VARY>(op, z, l, col, k, beta * q[l], zc);
      sig = fma(pc, qn, sig);
      p[l] = pc;
      q[l] = qn;
    }
  }
  double S, unused;
  if (grid_sum2<kSpmvThreads>(sig, 0.0, partials, &st->ticket_a, S, unused)) {
    st->last_sigma = S;
    if (!(S > 0.0) || !(S < INFINITY)) {
      st->alpha = 0.0;  // x keeps the iterate before this direction
      st->iters = st->it - 1;
      st->status = kStBreakdown;
      __threadfence();
      st->done = 1;
    } else {
      st->alpha = st->kappa_old / S;
    }
  }
}

// True when x is +0.0 (all bits zero) at the cell pair and at every point
// its stencil reads, so that A x is exactly zero there.
__device__ __forceinline__ bool x_is_zero2(const Op& op, const double* __restrict__ x,
                                           long long l, long long col, int k, double2 xc) {
  const int nz = op.nz;
  const Nbr nb = neighbours(op, col);
  unsigned long long bits = __double_as_longlong(xc.x) | __double_as_longlong(xc.y);
  if (k > 0) bits |= __double_as_longlong(x[l - 1]);
  if (k + 2 < nz) bits |= __double_as_longlong(x[l + 2]);
  const double2 e = ld2(x + nb.e * nz + k), w = ld2(x + nb.w * nz + k);
  const double2 n = ld2(x + nb.n * nz + k), s = ld2(x + nb.s * nz + k);
  bits |= __double_as_longlong(e.x) | __double_as_longlong(e.y) | __double_as_longlong(w.x) |
          __double_as_longlong(w.y) | __double_as_longlong(n.x) | __double_as_longlong(n.y) |
          __double_as_longlong(s.x) | __double_as_longlong(s.y);
  return bits == 0ull;
}

// MODE 0: y = A x.  MODE 1: r = b - A x, p = q = 0, and
// the scalar state of a new solve (alpha = 0, kappa_old = 1: the first sweeps
// then give p = z_0, q = A z_0).
template <bool VARY, bool VEC2, int MODE>
__global__ void __launch_bounds__(kSpmvThreads) k_stencil(Op op, DevState* st,
                                                          const double* __restrict__ x,
                                                          const double* __restrict__ b,
                                                          double* __restrict__ y,
                                                          double* __restrict__ p,
                                                          double* __restrict__ q, double rtol,
                                                          int maxit) {
  if (MODE == 1 && blockIdx.x == 0 && threadIdx.x == 0) {
    st->alpha = 0.0;
    st->beta = 0.0;
    st->kappa_old = 1.0;
    st->R0 = 0.0;
    st->rtol = rtol;
    st->last_sigma = st->last_kappa = st->last_R = 0.0;
    st->it = 0;
    st->status = kStOK;
    st->iters = 0;
    st->maxit = maxit;
    st->ticket_m = 0u;
    st->ticket_a = 0u;
    st->bar_count = 0u;
    st->dev_error = 0;
    st->done = 0;
  }
  const int nz = op.nz;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC2) {
    const long long np = op.n >> 1;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < np; g += stride) {
      const long long l = g << 1;
      const long long col = l / nz;
      const int k = (int)(l - col * nz);
      const double2 xc = ld2(x + l);
      double2 ax;
      if (MODE == 1 && x_is_zero2(op, x, l, col, k, xc)) {
        ax = make_double2(0.0, 0.0);  // A 0 = 0: the common zero initial guess costs no fp64
      } else {
        ax = stencil2<VARY>(op, x, l, col, k, make_double2(0.0, 0.0), xc);
      }
      if (MODE == 0) {
        st2(y + l, ax);
      } else {
        const double2 bv = ld2(b + l);
        st2(y + l, make_double2(bv.x - ax.x, bv.y - ax.y));
        st2(p + l, make_double2(0.0, 0.0));
        st2(q + l, make_double2(0.0, 0.0));
      }
    }
  } else {
    for (long long l = blockIdx.x * (long long)blockDim.x + threadIdx.x; l < op.n; l += stride) {
      const long long col = l / nz;
      const int k = (int)(l - col * nz);
      const double ax = stencil1<VARY>(op, x, l, col, k, 0.0, x[l]);
      if (MODE == 0) {
        y[l] = ax;
      } else {
        y[l] = b[l] - ax;
        p[l] = 0.0;
        q[l] = 0.0;
      }
    }
  }
}

// st->x0_nonzero |= (some value of x has a bit set); one atomic per warp that
// saw one.
__global__ void __launch_bounds__(256) k_x0_nonzero(const double* __restrict__ x, long long n,
                                                    DevState* st) {
  unsigned long long bits = 0ull;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    bits |= __double_as_longlong(x[i]);
  if (__any_sync(0xffffffffu, bits != 0ull) && (threadIdx.x & 31) == 0)
    atomicOr(&st->x0_nonzero, 1);
}

// Start of a solve in the row-tiled layout, one kernel: r = b - A x0 from the
// caller's column-contiguous b and x0, written row-tiled together with u = x0
// (and p = q = 0 with zero_pq: a solve whose first sweeps are the
// first-iteration variants reads neither), and the scalar state of a new
// solve (as k_stencil MODE 1).
// A block takes one tile of 32 columns and 32 levels: it reads along k
// (coalesced in the caller's layout), turns the 32 x 32 patch around in
// shared memory, and writes along the columns (coalesced in the solver's).
// Where x0 is +0.0 at a cell and at every point its stencil reads, r = b
// exactly and no fp64 work is done (the common zero initial guess).  With
// CHECKED, st->x0_nonzero == 0 says that all of x0 is +0.0: then neither x0
// nor its neighbours are read at all (r = b, u = 0).
template <bool VARY, bool CHECKED>
__global__ void __launch_bounds__(256) k_residual_tiled(Op op, DevState* st,
                                                        const double* __restrict__ x,
                                                        const double* __restrict__ b,
                                                        double* __restrict__ r_t,
                                                        double* __restrict__ u_t,
                                                        double* __restrict__ p_t,
                                                        double* __restrict__ q_t, double rtol,
                                                        int maxit, bool zero_pq) {
  const bool x_zero = CHECKED && st->x0_nonzero == 0;  // (the reset below leaves the flag)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    st->alpha = 0.0;
    st->beta = 0.0;
    st->kappa_old = 1.0;
    st->R0 = 0.0;
    st->rtol = rtol;
    st->last_sigma = st->last_kappa = st->last_R = 0.0;
    st->it = 0;
    st->status = kStOK;
    st->iters = 0;
    st->maxit = maxit;
    st->ticket_m = 0u;
    st->ticket_a = 0u;
    st->bar_count = 0u;
    st->dev_error = 0;
    st->done = 0;
  }
  __shared__ double sr[kTile][kTile + 1], sx[kTile][kTile + 1];
  const int nz = op.nz;
  const long long t = blockIdx.x;
  const int k0 = blockIdx.y * kTile;
  const int lane = threadIdx.x & 31, row = threadIdx.x >> 5;  // 8 rows of 32 threads
#pragma unroll
  for (int pass = 0; pass < kTile / 8; ++pass) {
    const int cl = row + 8 * pass, k = k0 + lane;
    const long long col = t * kTile + cl;
    double rv = 0.0, xv = 0.0;
    if (x_zero) {
      if (col < op.ncols && k < nz) rv = b[col * nz + k];
    } else if (col < op.ncols && k < nz) {
      const long long l = col * nz + k;
      xv = x[l];
      const Nbr nb = neighbours(op, col);
      unsigned long long bits = __double_as_longlong(xv);
      if (k > 0) bits |= __double_as_longlong(x[l - 1]);
      if (k + 1 < nz) bits |= __double_as_longlong(x[l + 1]);
      bits |= __double_as_longlong(x[nb.e * nz + k]) | __double_as_longlong(x[nb.w * nz + k]) |
              __double_as_longlong(x[nb.n * nz + k]) | __double_as_longlong(x[nb.s * nz + k]);
      rv = (bits == 0ull) ? b[l] : b[l] - stencil1<VARY>(op, x, l, col, k, 0.0, xv);
    }
    sr[lane][cl] = rv;
    sx[lane][cl] = xv;
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < kTile / 8; ++pass) {
    const int kk = row + 8 * pass, k = k0 + kk;
    if (k < nz) {
      const long long o = (t * nz + k) * kTile + lane;
      r_t[o] = sr[kk][lane];
      u_t[o] = sx[kk][lane];
      if (zero_pq) {
        p_t[o] = 0.0;
        q_t[o] = 0.0;
      }
    }
  }
}

template <bool VEC2>
__global__ void __launch_bounds__(kSpmvThreads) k_finalize(Op op, const DevState* st,
                                                           double* __restrict__ x,
                                                           const double* __restrict__ p) {
  const double alpha = st->alpha;
  if (alpha == 0.0) return;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (VEC2) {
    const long long np = op.n >> 1;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < np; g += stride) {
      double2 xv = ld2(x + 2 * g);
      const double2 pv = ld2(p + 2 * g);
      xv.x = fma(alpha, pv.x, xv.x);
      xv.y = fma(alpha, pv.y, xv.y);
      st2(x + 2 * g, xv);
    }
  } else {
    for (long long l = blockIdx.x * (long long)blockDim.x + threadIdx.x; l < op.n; l += stride)
      x[l] = fma(alpha, p[l], x[l]);
  }
}

// ------------------------------------------------------------- dispatch

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool staged(const Op& op) { return op.nz <= kMaxStagedNz; }
inline size_t staged_smem(const Op& op) { return 2u * kTile * (size_t)op.pz * sizeof(double); }

// Which preconditioner sweep a launch takes: 0 bulk-copy tile (nz even,
// 16-byte aligned vectors), 1 swizzled tile filled by scalar loads (odd nz or
// 8-byte aligned vectors), 2 unstaged (columns taller than the tile).
inline int precond_path(const Op& op, const double* r, const double* q, const double* z) {
  if (!staged(op)) return 2;
  const bool al = aligned16(r) && aligned16(z) && (!q || aligned16(q));
  return (op.nz % 2 == 0 && al) ? 0 : 1;
}

template <bool VARY, bool FUSED>
cudaError_t run_precond(const Op& op, DevState* st, double* r, const double* q, double* z,
                        double* partials, double* hist, int grid, cudaStream_t s) {
  switch (precond_path(op, r, q, z)) {
    case 0:
      if (op.fixed && op.nz == 128)
        k_precond_fixed<128, VARY, FUSED><<<grid, kTile, op.fixed_smem, s>>>(
            op, st, r, q, z, partials, hist);
      else if (op.fixed && op.nz == 64)
        k_precond_fixed<64, VARY, FUSED><<<grid, kTile, op.fixed_smem, s>>>(
            op, st, r, q, z, partials, hist);
      else if (op.fixed && op.nz == 32)
        k_precond_fixed<32, VARY, FUSED><<<grid, kTile, op.fixed_smem, s>>>(
            op, st, r, q, z, partials, hist);
      else if (op.nz % kChunk == 0)
        k_precond_stream<VARY, FUSED, true><<<grid, kTile, op.stream_smem, s>>>(
            op, st, r, q, z, partials, hist);
      else
        k_precond_stream<VARY, FUSED, false><<<grid, kTile, op.stream_smem, s>>>(
            op, st, r, q, z, partials, hist);
      break;
    case 1:
      k_precond_staged<VARY, FUSED><<<grid, kTile, staged_smem(op), s>>>(op, st, r, q, z,
                                                                         partials, hist);
      break;
    default:
      k_precond_direct<VARY, FUSED><<<grid, kTile, 0, s>>>(op, st, r, q, z, partials, hist);
  }
  return cudaGetLastError();
}

template <bool FUSED>
cudaError_t run_precond_any(const Op& op, DevState* st, double* r, const double* q, double* z,
                            double* partials, double* hist, int grid, cudaStream_t s) {
  return op.varying ? run_precond<true, FUSED>(op, st, r, q, z, partials, hist, grid, s)
                    : run_precond<false, FUSED>(op, st, r, q, z, partials, hist, grid, s);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// ------------------------------------------------------------- launchers

cudaError_t prepare_kernels(const Op& op) {
  if (!staged(op)) return cudaSuccess;
  {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    size_t stat = 0;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k_precond_stream<true, true, true>) == cudaSuccess)
      stat = std::max(stat, fa.sharedSizeBytes);
    if (cudaFuncGetAttributes(&fa, k_precond_stream<false, true, false>) == cudaSuccess)
      stat = std::max(stat, fa.sharedSizeBytes);
    g_max_stream_smem = optin - (int)stat;
  }
  const int kMaxStreamSmem = g_max_stream_smem;
  const size_t b = staged_smem(op);
  cudaError_t e = cudaSuccess;
  cudaError_t r;
#define PCG_SET(V, F)                                             \
  r = set_smem(k_precond_staged<V, F>, b);                        \
  if (r != cudaSuccess) e = r;                                    \
  r = set_smem(k_precond_fixed<128, V, F>, kMaxStreamSmem);       \
  if (r != cudaSuccess) e = r;                                    \
  r = set_smem(k_precond_fixed<64, V, F>, kMaxStreamSmem);        \
  if (r != cudaSuccess) e = r;                                    \
  r = set_smem(k_precond_fixed<32, V, F>, kMaxStreamSmem);        \
  if (r != cudaSuccess) e = r;                                    \
  r = set_smem(k_precond_stream<V, F, true>, kMaxStreamSmem);     \
  if (r != cudaSuccess) e = r;                                    \
  r = set_smem(k_precond_stream<V, F, false>, kMaxStreamSmem);    \
  if (r != cudaSuccess) e = r;
  PCG_SET(false, false) PCG_SET(false, true) PCG_SET(true, false) PCG_SET(true, true)
#undef PCG_SET
  return e;
}

// The streaming sweep runs one warp per block.  Each of the four
// sub-partitions of an SM has its own fp64 unit, so the launch asks for
// enough shared memory that the resident warps per SM are a multiple of four
// (4 at nz = 128, 8 for short columns): a fifth warp would share a
// sub-partition with another and, under the static tile assignment, set the
// pace for the whole grid.
int grid_precond(Op& op, int num_sms) {
  int per_sm = 0;
  cudaError_t e = cudaSuccess;
  op.stream_smem = (int)stream_smem_bytes<true>(op.pt);
  op.fixed_smem = (int)fixed_smem_bytes<true>();
  if (op.fixed) {
    // Two warps per sub-partition: eight per SM (the register file allows up
    // to ten); the shared-memory request is padded so that no ninth fits.
    int dev = 0, smem_sm = 0, reserved = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    auto occ = [&](int bytes) {
      int b = 0;
      cudaError_t r = cudaErrorInvalidValue;
#define PCG_OCC(NZ)                                                                         \
  if (op.nz == NZ)                                                                          \
    r = op.varying                                                                          \
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_precond_fixed<NZ, true, true>, \
                                                            kTile, bytes)                   \
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(                                \
                  &b, k_precond_fixed<NZ, false, true>, kTile, bytes);
      PCG_OCC(128) PCG_OCC(64) PCG_OCC(32)
#undef PCG_OCC
      return r == cudaSuccess ? b : 0;
    };
    per_sm = occ(op.fixed_smem);
    if (per_sm > 4 && per_sm % 4 != 0) {
      const int target = per_sm / 4 * 4;
      const int padded = smem_sm / target - reserved - 256;
      if (padded > op.fixed_smem && padded <= g_max_stream_smem && occ(padded) == target) {
        op.fixed_smem = padded;
        per_sm = target;
      }
    }
  } else if (staged(op)) {
    int dev = 0, smem_sm = 0, reserved = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    auto occ = [&](int bytes) {
      int b = 0;
      cudaError_t r = op.varying ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                       &b, k_precond_stream<true, true, true>, kTile, bytes)
                                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                       &b, k_precond_stream<false, true, true>, kTile, bytes);
      return r == cudaSuccess ? b : 0;
    };
    per_sm = occ(op.stream_smem);
    if (per_sm > 4 && per_sm % 4 != 0) {
      const int target = per_sm / 4 * 4;
      const int padded = smem_sm / target - reserved - 256;
      if (padded > op.stream_smem && padded <= g_max_stream_smem && occ(padded) == target) {
        op.stream_smem = padded;
        per_sm = target;
      }
    }
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_precond_direct<false, true>,
                                                      kTile, 0);
  }
  if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  long long g = (long long)per_sm * num_sms;
  if (g > op.ntiles) g = op.ntiles;
  return (int)(g < 1 ? 1 : g);
}

int grid_spmv(const Op& op, int num_sms) {
  int per_sm = 0;
  cudaError_t e = op.varying ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                   &per_sm, k_spmv_fused<true, true, false>, kSpmvThreads, 0)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                   &per_sm, k_spmv_fused<false, true, false>, kSpmvThreads, 0);
  if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  long long g = (long long)per_sm * num_sms;
  const long long work = (op.n + 2 * kSpmvThreads - 1) / (2 * kSpmvThreads);
  if (g > work) g = work;
  return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_residual(const Op& op, DevState* st, const double* b, const double* x,
                            double* r, double* p, double* q, double rtol, int maxit, int grid,
                            cudaStream_t s) {
  const bool v2 = (op.nz % 2 == 0) && aligned16(b) && aligned16(x) && aligned16(r) &&
                  aligned16(p) && aligned16(q);
  if (op.varying) {
    if (v2) k_stencil<true, true, 1><<<grid, kSpmvThreads, 0, s>>>(op, st, x, b, r, p, q, rtol, maxit);
    else k_stencil<true, false, 1><<<grid, kSpmvThreads, 0, s>>>(op, st, x, b, r, p, q, rtol, maxit);
  } else {
    if (v2) k_stencil<false, true, 1><<<grid, kSpmvThreads, 0, s>>>(op, st, x, b, r, p, q, rtol, maxit);
    else k_stencil<false, false, 1><<<grid, kSpmvThreads, 0, s>>>(op, st, x, b, r, p, q, rtol, maxit);
  }
  return cudaGetLastError();
}

cudaError_t launch_residual_tiled(const Op& op, DevState* st, const double* b, const double* x,
                                  double* r_t, double* u_t, double* p_t, double* q_t, double rtol,
                                  int maxit, bool x0_checked, cudaStream_t s, bool zero_pq) {
  const dim3 g((unsigned)op.ntiles, (unsigned)((op.nz + kTile - 1) / kTile));
#define PCG_RES(VY, CK) \
  k_residual_tiled<VY, CK><<<g, 256, 0, s>>>(op, st, x, b, r_t, u_t, p_t, q_t, rtol, maxit, \
                                             zero_pq)
  if (op.varying) {
    if (x0_checked) PCG_RES(true, true); else PCG_RES(true, false);
  } else {
    if (x0_checked) PCG_RES(false, true); else PCG_RES(false, false);
  }
#undef PCG_RES
  return cudaGetLastError();
}

cudaError_t launch_x0_nonzero(const double* x, long long n, DevState* st, int num_sms,
                              cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(&st->x0_nonzero, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  const long long g = std::max<long long>(1, std::min<long long>((n + 1023) / 1024,
                                                                 16LL * num_sms));
  k_x0_nonzero<<<(int)g, 256, 0, s>>>(x, n, st);
  return cudaGetLastError();
}

cudaError_t launch_apply(const Op& op, const double* x, double* y, int grid, cudaStream_t s) {
  const bool v2 = (op.nz % 2 == 0) && aligned16(x) && aligned16(y);
  if (op.varying) {
    if (v2) k_stencil<true, true, 0><<<grid, kSpmvThreads, 0, s>>>(op, nullptr, x, nullptr, y, nullptr, nullptr, 0.0, 0);
    else k_stencil<true, false, 0><<<grid, kSpmvThreads, 0, s>>>(op, nullptr, x, nullptr, y, nullptr, nullptr, 0.0, 0);
  } else {
    if (v2) k_stencil<false, true, 0><<<grid, kSpmvThreads, 0, s>>>(op, nullptr, x, nullptr, y, nullptr, nullptr, 0.0, 0);
    else k_stencil<false, false, 0><<<grid, kSpmvThreads, 0, s>>>(op, nullptr, x, nullptr, y, nullptr, nullptr, 0.0, 0);
  }
  return cudaGetLastError();
}

cudaError_t launch_precond(const Op& op, DevState* st, const double* r, double* z, int grid,
                           cudaStream_t s) {
  return run_precond_any<false>(op, st, const_cast<double*>(r), nullptr, z, nullptr, nullptr,
                                grid, s);
}

cudaError_t launch_precond_fused(const Op& op, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s) {
  return run_precond_any<true>(op, st, r, q, z, partials, hist, grid, s);
}

cudaError_t launch_spmv_fused(const Op& op, DevState* st, const double* z, const double* r,
                              double* u, double* p, double* q, double* partials, int grid,
                              cudaStream_t s) {
  const bool v2 = (op.nz % 2 == 0) && aligned16(z) && aligned16(r) && aligned16(u) &&
                  aligned16(p) && aligned16(q);
  const bool rs = op.az_resid != 0;
#define PCG_SPMV(VY, V2, RS) \
  k_spmv_fused<VY, V2, RS><<<grid, kSpmvThreads, 0, s>>>(op, st, z, r, u, p, q, partials)
  if (op.varying) {
    if (rs) {
      if (v2) PCG_SPMV(true, true, true); else PCG_SPMV(true, false, true);
    } else {
      if (v2) PCG_SPMV(true, true, false); else PCG_SPMV(true, false, false);
    }
  } else {
    if (rs) {
      if (v2) PCG_SPMV(false, true, true); else PCG_SPMV(false, false, true);
    } else {
      if (v2) PCG_SPMV(false, true, false); else PCG_SPMV(false, false, false);
    }
  }
#undef PCG_SPMV
  return cudaGetLastError();
}

cudaError_t launch_finalize(const Op& op, const DevState* st, double* x, const double* p,
                            int grid, cudaStream_t s) {
  if (aligned16(x) && aligned16(p) && (op.n % 2 == 0))
    k_finalize<true><<<grid, kSpmvThreads, 0, s>>>(op, st, x, p);
  else
    k_finalize<false><<<grid, kSpmvThreads, 0, s>>>(op, st, x, p);
  return cudaGetLastError();
}

}  // namespace pcg
