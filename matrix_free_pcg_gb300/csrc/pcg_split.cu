// Substructured (parallel-in-k) column solve for the preconditioner sweep,
// row-tiled layout.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 6.1 (the substructuring method for the vertical tridiagonal
// systems, after Toselli and Widlund) applied to the column blocks of M,
// eq. (19), inside the fused sweep of Appendix A, Algorithm 3.
//
// Each column of nz levels is cut into P blocks by P-1 interface levels
// (block i: levels s_i .. s_i+m_i-1; interface i after it, at s_i+m_i).
// With the block interiors B_i eliminated first, M z = r splits into
//   1. y_i = T_i^{-1} r_i for every block (independent: one warp per block);
//   2. a tridiagonal system of size P-1 for the interface values (Schur
//      complement S = T_gg - sum_i T_gi T_i^{-1} T_ig), per column;
//   3. z_i = y_i + t_L z_left a_i + t_R z_right b_i, with the "spikes"
//      a_i = T_i^{-1} e_first, b_i = T_i^{-1} e_last and the couplings t_L,
//      t_R of the block's end levels to its interface neighbours.
// Every matrix-dependent quantity (LDL^T factors of each T_i, the scaled
// spikes, the LDL^T factors of S) is formed once per operator by the set-up
// kernels below.  In exact arithmetic the result is M^{-1} r; the rounding
// differs from a single Thomas sweep by a few units of cond(T) * eps.
//
// <r, z> needs no extra pass: per block, <r_i, z_i> = <r_i, y_i>
// + t_L z_left (y_i)_first + t_R z_right (y_i)_last (T_i symmetric), and
// <r_i, y_i> = sum_k y'_k w_k from the block's forward elimination, as in the
// single-sweep kernel; the interface levels add r_g z_g.
//
// Layout: tables and vectors row-tiled, cell (column c, level k) at
// (c/32*nz + k)*32 + c%32; per-column interface data at
// ((c/32)*(P-1) + j)*32 + c%32; block corners at ((c/32)*P + i)*4*32 + ...
#include <algorithm>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"

namespace pcg {
namespace {

// Block i of P in a column of nz levels: first level s, interior length m.
__host__ __device__ __forceinline__ void split_block(int nz, int P, int i, int& s, int& m) {
  const int base = (nz - (P - 1)) / P, rem = (nz - (P - 1)) % P;
  s = i * (base + 1) + min(i, rem);
  m = base + (i < rem ? 1 : 0);
}

// Full diagonal of M at level k of a column whose four face values sum to sf.
__device__ __forceinline__ double split_diag(const Op& op, int k, double sf) {
  const int nz = op.nz;
  return op.varying ? op.lev[LV_DIAG * nz + k] + op.lev[LV_H * nz + k] * sf
                    : op.lev[LV_DIAG * nz + k];
}

__device__ __forceinline__ double face_sum(const Op& op, long long col) {
  if (!op.varying) return 0.0;
  const Nbr nb = neighbours(op, col);
  return op.faceE[col] + op.faceE[nb.w] + op.faceN[col] + op.faceN[nb.s];
}

// Set-up 1: one thread per (column, block).  LDL^T of the block,
// D_k = diag_k - T_{k-1/2} (T_{k-1/2}/D_{k-1}) from its first level, stored as
// nphi_k = T_{k+1/2}/D_k (0 at the block's last level) and 1/D_k; the scaled
// spikes t_L a and t_R b; the corners a_first, a_last, b_first, b_last.
__global__ void k_split_blocks(Op op, int P, DevState* st, double* __restrict__ nphi,
                               double* __restrict__ invd, double* __restrict__ ta,
                               double* __restrict__ tb, double* __restrict__ corners) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  const long long total = op.ntiles * P * kTile;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(g % kTile);
    const int i = (int)((g / kTile) % P);
    const long long t = g / ((long long)kTile * P);
    const long long col = t * kTile + lane;
    if (col >= op.ncols) continue;
    int s, m;
    split_block(nz, P, i, s, m);
    const double sf = face_sum(op, col);
    const long long base = t * nz * kTile + lane;
    auto at = [&](int k) { return base + (long long)k * kTile; };
    int bad = 0;
    double np = 0.0;
    for (int k = s; k < s + m; ++k) {
      const double D = split_diag(op, k, sf) - (k > s ? lev[LV_TDN * nz + k] * np : 0.0);
      if (!(D > 0.0)) bad = 1;
      invd[at(k)] = 1.0 / D;
      np = (k < s + m - 1) ? lev[LV_TUP * nz + k] / D : 0.0;
      nphi[at(k)] = np;
    }
    // a = T_i^{-1} e_first: forward y'_k = nphi_{k-1} y'_{k-1} from 1, w = y'/D,
    // back a_k = w_k + nphi_k a_{k+1}.  b = T_i^{-1} e_last: w nonzero only at
    // the last level, back b_k = nphi_k b_{k+1}.
    double yp = 1.0;
    for (int k = s; k < s + m; ++k) {
      if (k > s) yp *= nphi[at(k - 1)];
      ta[at(k)] = yp * invd[at(k)];
    }
    double a = ta[at(s + m - 1)], b = invd[at(s + m - 1)];
    tb[at(s + m - 1)] = b;
    for (int k = s + m - 2; k >= s; --k) {
      a = ta[at(k)] + nphi[at(k)] * a;
      b = nphi[at(k)] * b;
      ta[at(k)] = a;
      tb[at(k)] = b;
    }
    double* cr = corners + ((t * P + i) * 4) * kTile + lane;
    cr[0] = ta[at(s)];
    cr[kTile] = ta[at(s + m - 1)];
    cr[2 * kTile] = tb[at(s)];
    cr[3 * kTile] = tb[at(s + m - 1)];
    const double tL = (i > 0) ? lev[LV_TDN * nz + s] : 0.0;            // T_{s-1/2}
    const double tR = (i < P - 1) ? lev[LV_TUP * nz + s + m - 1] : 0.0;  // T_{s+m-1/2}
    for (int k = s; k < s + m; ++k) {
      ta[at(k)] *= tL;
      tb[at(k)] *= tR;
    }
    if (bad) st->setup_error = 1;
  }
}

// Set-up 2: one thread per column.  Schur complement on the interface levels
// g_j = s_j + m_j (j = 0..P-2):
//   S_jj     = diag_g - T_{g-1/2}^2 (T_j^{-1})_{last,last} - T_{g+1/2}^2 (T_{j+1}^{-1})_{first,first}
//   S_j,j+1  = -T_{g_j+1/2} T_{g_{j+1}-1/2} (T_{j+1}^{-1})_{first,last}
// and its LDL^T factors, stored as 1/DS_j and nphiS_j = -S_j,j+1 / DS_j.
__global__ void k_split_schur(Op op, int P, DevState* st, const double* __restrict__ corners,
                              double* __restrict__ invdS, double* __restrict__ nphiS) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  for (long long col = blockIdx.x * (long long)blockDim.x + threadIdx.x; col < op.ncols;
       col += (long long)gridDim.x * blockDim.x) {
    const long long t = col / kTile;
    const int lane = (int)(col - t * kTile);
    const double sf = face_sum(op, col);
    auto corner = [&](int i, int c) { return corners[((t * P + i) * 4 + c) * kTile + lane]; };
    double Dprev = 0.0, Sprev = 0.0;
    int bad = 0;
    for (int j = 0; j < P - 1; ++j) {
      int sj, mj, s1, m1;
      split_block(nz, P, j, sj, mj);
      split_block(nz, P, j + 1, s1, m1);
      const int g = sj + mj;
      const double tdn = lev[LV_TDN * nz + g], tup = lev[LV_TUP * nz + g];
      const double Sd = split_diag(op, g, sf) - tdn * tdn * corner(j, 3) - tup * tup * corner(j + 1, 0);
      const double So = (j + 1 < P - 1) ? -tup * lev[LV_TUP * nz + s1 + m1 - 1] * corner(j + 1, 2) : 0.0;
      const double D = Sd - (j > 0 ? Sprev * Sprev / Dprev : 0.0);
      if (!(D > 0.0)) bad = 1;
      const long long o = (t * (P - 1) + j) * kTile + lane;
      invdS[o] = 1.0 / D;
      nphiS[o] = -So / D;
      Dprev = D;
      Sprev = So;
    }
    if (bad) st->setup_error = 1;
  }
}

// Algorithm 3 sweep with the substructured column solve: a block of P warps
// per tile of 32 columns, warp i on block i of every column.  The shared
// tiles W and N (nz x 32 each, level-major) hold w (then y) and the block's
// nphi; yF, yL, rg and zg exchange the block ends, the interface residuals
// and the interface solution between the warps.  Every global load of a
// pass is independent of its recurrence, so operands arrive kSpChunk levels
// at a time, one chunk ahead of their use (4 levels for 16 warps per block,
// whose threads may hold at most 128 registers).
template <int P>
__global__ void __launch_bounds__(P * 32) k_precond_split(Op op, DevState* st,
                                                          double* __restrict__ r,
                                                          const double* __restrict__ q,
                                                          double* __restrict__ z,
                                                          double* __restrict__ partials,
                                                          double* __restrict__ hist) {
  constexpr int kSpChunk = 4;
  extern __shared__ double smem[];
  if (ld_done(st)) return;
  const int lane = threadIdx.x & 31, i = threadIdx.x >> 5;
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  double* Wt = smem;               // nz * 32: w, then y
  double* Nt = Wt + nz * kTile;    // nz * 32: the block's nphi
  double* yF = Nt + nz * kTile;    // P * 32: first level of y_i
  double* yL = yF + P * kTile;     // P * 32: last level of y_i
  double* rg = yL + P * kTile;     // P * 32: r* at interface i
  double* zg = rg + P * kTile;     // (P+1) * 32: z at interface i-1 (zg[0] = zg[P] = 0)
  const double nalpha = -st->alpha;
  const uint64_t stream = l2_stream();
  int s, m;
  split_block(nz, P, i, s, m);
  const int e = s + m;  // one past the block's last level
  const double tL = (i > 0) ? lev[LV_TDN * nz + s] : 0.0;
  const double tR = (i < P - 1) ? lev[LV_TUP * nz + e - 1] : 0.0;
  double accR = 0.0, accK = 0.0;
  for (long long t = blockIdx.x; t < op.ntiles; t += gridDim.x) {
    const bool act = t * kTile + lane < op.ncols;
    const long long base = t * nz * kTile + lane;
    // ---- 1. r* = r - alpha q and the block solve y_i = T_i^{-1} r*_i
    if (act) {
      double cr[kSpChunk], cq[kSpChunk], ci[kSpChunk], cn[kSpChunk];
#pragma unroll
      for (int j = 0; j < kSpChunk; ++j) {
        const long long o = base + (long long)(s + j) * kTile;
        const bool in = s + j < e;
        cr[j] = in ? ld_hint(r + o, stream) : 0.0;
        cq[j] = in ? ld_hint(q + o, stream) : 0.0;
        ci[j] = in ? ld_hint(op.sp_invd + o, stream) : 0.0;
        cn[j] = in ? ld_hint(op.sp_nphi + o, stream) : 0.0;
      }
      double rgi = 0.0;
      if (i < P - 1) {  // interface level after the block
        const long long o = base + (long long)e * kTile;
        rgi = fma(nalpha, q[o], r[o]);
      }
      double yp = 0.0, np = 0.0;
#pragma unroll 1
      for (int k0 = s; k0 < e; k0 += kSpChunk) {
        double nr[kSpChunk], nq[kSpChunk], ni[kSpChunk], nn[kSpChunk];
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          const long long o = base + (long long)(k0 + kSpChunk + j) * kTile;
          const bool in = k0 + kSpChunk + j < e;
          nr[j] = in ? ld_hint(r + o, stream) : 0.0;
          nq[j] = in ? ld_hint(q + o, stream) : 0.0;
          ni[j] = in ? ld_hint(op.sp_invd + o, stream) : 0.0;
          nn[j] = in ? ld_hint(op.sp_nphi + o, stream) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          const int k = k0 + j;
          if (k < e) {
            const double rk = fma(nalpha, cq[j], cr[j]);
            accR = fma(rk, rk, accR);
            st_hint(r + base + (long long)k * kTile, rk, stream);
            yp = fma(np, yp, rk);
            const double w = yp * ci[j];
            accK = fma(yp, w, accK);
            Wt[k * kTile + lane] = w;
            Nt[k * kTile + lane] = cn[j];
            np = cn[j];
          }
        }
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          cr[j] = nr[j];
          cq[j] = nq[j];
          ci[j] = ni[j];
          cn[j] = nn[j];
        }
      }
      double yy = Wt[(e - 1) * kTile + lane];
      yL[i * kTile + lane] = yy;
      for (int k = e - 2; k >= s; --k) {
        yy = fma(Nt[k * kTile + lane], yy, Wt[k * kTile + lane]);
        Wt[k * kTile + lane] = yy;
      }
      yF[i * kTile + lane] = yy;
      if (i < P - 1) {
        accR = fma(rgi, rgi, accR);
        r[base + (long long)e * kTile] = rgi;
        rg[i * kTile + lane] = rgi;
      }
    }
    __syncthreads();
    // ---- 2. interface system (warp 0, one lane per column)
    if (i == 0 && act) {
      const long long sb = t * (P - 1) * kTile + lane;
      double ys = 0.0, npS = 0.0;
      int sj = 0, mj = 0;
      for (int j = 0; j < P - 1; ++j) {
        split_block(nz, P, j, sj, mj);
        const int g = sj + mj;
        const double rhs = fma(lev[LV_TUP * nz + g], yF[(j + 1) * kTile + lane],
                               fma(lev[LV_TDN * nz + g], yL[j * kTile + lane], rg[j * kTile + lane]));
        ys = fma(npS, ys, rhs);
        zg[(j + 1) * kTile + lane] = ys * op.sp_invdS[sb + (long long)j * kTile];
        npS = op.sp_nphiS[sb + (long long)j * kTile];
      }
      double zz = zg[(P - 1) * kTile + lane];
      accK = fma(rg[(P - 2) * kTile + lane], zz, accK);
      for (int j = P - 3; j >= 0; --j) {
        zz = fma(op.sp_nphiS[sb + (long long)j * kTile], zz, zg[(j + 1) * kTile + lane]);
        zg[(j + 1) * kTile + lane] = zz;
        accK = fma(rg[j * kTile + lane], zz, accK);
      }
      zg[lane] = 0.0;
      zg[P * kTile + lane] = 0.0;
    }
    __syncthreads();
    // ---- 3. z_i = y_i + (t_L a_i) z_left + (t_R b_i) z_right
    if (act) {
      const double zl = zg[i * kTile + lane], zr = zg[(i + 1) * kTile + lane];
      double ca[kSpChunk], cb[kSpChunk];
#pragma unroll
      for (int j = 0; j < kSpChunk; ++j) {
        const long long o = base + (long long)(s + j) * kTile;
        const bool in = s + j < e;
        ca[j] = in ? ld_hint(op.sp_ta + o, stream) : 0.0;
        cb[j] = in ? ld_hint(op.sp_tb + o, stream) : 0.0;
      }
#pragma unroll 1
      for (int k0 = s; k0 < e; k0 += kSpChunk) {
        double na[kSpChunk], nb2[kSpChunk];
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          const long long o = base + (long long)(k0 + kSpChunk + j) * kTile;
          const bool in = k0 + kSpChunk + j < e;
          na[j] = in ? ld_hint(op.sp_ta + o, stream) : 0.0;
          nb2[j] = in ? ld_hint(op.sp_tb + o, stream) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          const int k = k0 + j;
          if (k < e)
            st_hint(z + base + (long long)k * kTile,
                    fma(cb[j], zr, fma(ca[j], zl, Wt[k * kTile + lane])), stream);
        }
#pragma unroll
        for (int j = 0; j < kSpChunk; ++j) {
          ca[j] = na[j];
          cb[j] = nb2[j];
        }
      }
      accK = fma(tL * zl, yF[i * kTile + lane], accK);
      accK = fma(tR * zr, yL[i * kTile + lane], accK);
      if (i < P - 1) z[base + (long long)e * kTile] = zr;
    }
    __syncthreads();  // the shared tiles are refilled for the next tile
  }
  double R, K;
  if (grid_sum2<P * 32>(accR, accK, partials, &st->ticket_m, R, K))
    finish_precond_sweep(st, R, K, hist);
}

template <int P>
cudaError_t run_split(const Op& op, DevState* st, double* r, const double* q, double* z,
                      double* partials, double* hist, int grid, cudaStream_t s) {
  k_precond_split<P><<<grid, P * 32, split_smem_bytes(op.nz, P), s>>>(op, st, r, q, z, partials,
                                                                      hist);
  return cudaGetLastError();
}

template <int P>
int split_grid_for(const Op& op, int num_sms) {
  const size_t smem = split_smem_bytes(op.nz, P);
  // a refused size (columns too tall for the shared tiles) is an answer, not
  // an error: clear it so that no later launch check reports it
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k_precond_split<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int a = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_precond_split<P>, P * 32, smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (a < 1) return 0;
  long long g = (long long)a * num_sms;
  if (g > op.ntiles) g = op.ntiles;
  return (int)std::max<long long>(g, 1);
}

}  // namespace

size_t split_smem_bytes(int nz, int P) {
  return sizeof(double) * (2 * (size_t)nz * kTile + (size_t)(4 * P + 1) * kTile);
}

bool split_valid(int nz, int P) {
  return (P == 2 || P == 4 || P == 8 || P == 16) && nz >= 2 * P - 1;
}

int split_grid(const Op& op, int P, int num_sms) {
  switch (P) {
    case 2: return split_grid_for<2>(op, num_sms);
    case 4: return split_grid_for<4>(op, num_sms);
    case 8: return split_grid_for<8>(op, num_sms);
    case 16: return split_grid_for<16>(op, num_sms);
    default: return 0;
  }
}

cudaError_t launch_split_setup(const Op& op, int P, DevState* st, cudaStream_t s) {
  const long long total = op.ntiles * P * kTile;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  blocks = std::min<long long>(blocks, 1 << 20);
  k_split_blocks<<<(int)blocks, threads, 0, s>>>(op, P, st, op.sp_nphi, op.sp_invd, op.sp_ta,
                                                 op.sp_tb, op.sp_corners);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  blocks = std::min<long long>((op.ncols + threads - 1) / threads, 1 << 20);
  k_split_schur<<<(int)blocks, threads, 0, s>>>(op, P, st, op.sp_corners, op.sp_invdS,
                                                op.sp_nphiS);
  return cudaGetLastError();
}

cudaError_t launch_precond_split(const Op& op, int P, DevState* st, double* r, const double* q,
                                 double* z, double* partials, double* hist, int grid,
                                 cudaStream_t s) {
  switch (P) {
    case 2: return run_split<2>(op, st, r, q, z, partials, hist, grid, s);
    case 4: return run_split<4>(op, st, r, q, z, partials, hist, grid, s);
    case 8: return run_split<8>(op, st, r, q, z, partials, hist, grid, s);
    case 16: return run_split<16>(op, st, r, q, z, partials, hist, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pcg
