// Cluster-resident solve loop for grids small enough to live in the shared
// memory of one thread-block cluster: every iteration of Algorithm 1, with
// every vector of the solve on chip.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 4.3 Algorithm 1 (loop), Appendix A Algorithms 2 and 3 (sweeps),
// with A z formed as r + (A - M) z from the z of M z = r.
//
// The C CTAs of one cluster own the row-tiled tiles round-robin (tile t on
// CTA t % C, slot t / C) and hold r, z, p, q, u and, for an a_h field, the
// Thomas factors and the horizontal weights of their tiles in shared memory.
// The preconditioner sweep touches only a CTA's own tiles; the stencil sweep
// reads the horizontal neighbours' z (and weights) from the owning CTA's
// shared memory through the cluster's distributed shared memory.  Each CTA
// writes its partial sums into a slot of every CTA's shared memory, so after
// one cluster barrier every CTA adds the same numbers in the same order and
// takes the same scalar decisions.  Two cluster barriers per iteration: the
// hardware barrier replaces the grid barrier through global memory of the
// persistent loop, and nothing polls a flag.
#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"

namespace cg = cooperative_groups;

namespace pcg {
namespace {

constexpr int kClThreads = 256;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClMaxCtas = 16;

// Shared-memory arrays per tile slot, in this order.
enum { CA_R = 0, CA_Z, CA_P, CA_Q, CA_U, CA_NPHI, CA_INVD, CA_WE, CA_WN, CA_COUNT };

// Offset (in doubles) of array a, slot j, level k, lane of a CTA's shared block.
__device__ __forceinline__ int cl_off(int a, int j, int k, int lane, int slots, int nz) {
  return ((a * slots + j) * nz + k) * kTile + lane;
}

// Block sums of NV values in a fixed order, written by thread 0 into slot
// `rank` of array `slot` (NV doubles per CTA) on every CTA of the cluster.
// Only the warps that had work in the sweep reduce with shuffles; the others
// contribute exact zeros without fp64 work (an fp64 warp instruction holds a
// sub-partition's fp64 pipe for 64 cycles whether its values are zero or not),
// and warp 0 adds the warp totals in a shuffle tree.
template <int NV>
__device__ __forceinline__ void cl_publish(cg::cluster_group& cluster, const double (&v)[NV],
                                           bool warp_busy, double* slot, int C) {
  __shared__ double sw[NV][kClWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const double s = warp_busy ? warp_sum(v[j]) : 0.0;
    if (lane == 0) sw[j][w] = s;
  }
  __syncthreads();
  if (w == 0) {
    double tot[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double a = (lane < kClWarps) ? sw[j][lane] : 0.0;
#pragma unroll
      for (int o = kClWarps / 2; o > 0; o >>= 1) a += __shfl_down_sync(0xffffffffu, a, o);
      tot[j] = a;
    }
    if (lane == 0) {
      const unsigned rank = cluster.block_rank();
      for (int r = 0; r < C; ++r) {
        double* remote = cluster.map_shared_rank(slot, r);
#pragma unroll
        for (int j = 0; j < NV; ++j) remote[NV * rank + j] = tot[j];
      }
    }
  }
}

// The cluster totals of published values, in rank order.
template <int NV>
__device__ __forceinline__ void cl_totals(const double* slot, int C, double (&t)[NV]) {
#pragma unroll
  for (int j = 0; j < NV; ++j) t[j] = 0.0;
  for (int r = 0; r < C; ++r) {
#pragma unroll
    for (int j = 0; j < NV; ++j) t[j] += slot[NV * r + j];
  }
}

template <bool VARY>
__global__ void __launch_bounds__(kClThreads, 1) k_pcg_cluster(Op op, DevState* st,
                                                            double* __restrict__ r_g,
                                                            double* __restrict__ u_g,
                                                            double* __restrict__ p_g,
                                                            double* __restrict__ hist,
                                                            int slots) {
  extern __shared__ double sm[];
  __shared__ double slotM[2 * kClMaxCtas], slotA[2 * kClMaxCtas];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int nz = op.nz;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const double* __restrict__ lev = op.lev;

  // ---- load the own tiles: r (from the start of the solve), u = x0,
  // p = q = 0, and for a field the factors and the weights
  for (int j = 0; j < slots; ++j) {
    const long long t = (long long)j * C + rank;
    for (int e = threadIdx.x; e < nz * kTile; e += kClThreads) {
      const int k = e / kTile, l = e - k * kTile;
      const bool in = t < op.ntiles && t * kTile + l < op.ncols;
      const long long g = (t * nz + k) * kTile + l;
      sm[cl_off(CA_R, j, k, l, slots, nz)] = in ? r_g[g] : 0.0;
      sm[cl_off(CA_Z, j, k, l, slots, nz)] = 0.0;
      sm[cl_off(CA_P, j, k, l, slots, nz)] = 0.0;
      sm[cl_off(CA_Q, j, k, l, slots, nz)] = 0.0;
      sm[cl_off(CA_U, j, k, l, slots, nz)] = in ? u_g[g] : 0.0;
      if (VARY) {
        sm[cl_off(CA_NPHI, j, k, l, slots, nz)] = in ? op.tnphi[g] : 0.0;
        sm[cl_off(CA_INVD, j, k, l, slots, nz)] = in ? op.tinvd[g] : 0.0;
        sm[cl_off(CA_WE, j, k, l, slots, nz)] = in ? op.cwE_t[g] : 0.0;
        sm[cl_off(CA_WN, j, k, l, slots, nz)] = in ? op.cwN_t[g] : 0.0;
      }
    }
  }
  cluster.sync();

  // The scalar step of every iteration is taken by thread 0 of each CTA (from
  // the same published numbers in the same order, so every CTA decides
  // alike); the other threads get alpha, beta and the stop flag through
  // shared memory.
  __shared__ double sh_alpha, sh_beta;
  __shared__ int sh_done;
  const double rtol = st->rtol;
  const int maxit = st->maxit;
  double alpha = 0.0, beta = 0.0, kappa_old = 1.0, R0 = 0.0, R = 0.0, K = 0.0, S = 0.0;
  int it = 0, iters = 0, status = kStOK;  // (thread 0's)
  const int segs = (slots >= kClWarps) ? 1 : kClWarps / slots;  // level segments per slot
  const int seglen = (nz + segs - 1) / segs;
  for (;;) {
    // ---- Algorithm 3 sweep on the own tiles: one warp per tile slot
    double accR = 0.0, accK = 0.0;
    const bool busyM = warp < slots && (long long)warp * C + rank < op.ntiles;
    for (int j = warp; j < slots; j += kClWarps) {
      const long long t = (long long)j * C + rank;
      if (t >= op.ntiles || t * kTile + lane >= op.ncols) continue;
      double y = 0.0, nprev = 0.0, w = 0.0;
      for (int k = 0; k < nz; ++k) {
        double& rk_s = sm[cl_off(CA_R, j, k, lane, slots, nz)];
        const double rk = fma(-alpha, sm[cl_off(CA_Q, j, k, lane, slots, nz)], rk_s);
        rk_s = rk;
        accR = fma(rk, rk, accR);
        y = fma(nprev, y, rk);
        w = y * (VARY ? sm[cl_off(CA_INVD, j, k, lane, slots, nz)] : lev[LV_INVD * nz + k]);
        accK = fma(y, w, accK);
        sm[cl_off(CA_Z, j, k, lane, slots, nz)] = w;
        nprev = VARY ? sm[cl_off(CA_NPHI, j, k, lane, slots, nz)] : lev[LV_NPHI * nz + k];
      }
      double zz = w;
      for (int k = nz - 2; k >= 0; --k) {
        const double nk = VARY ? sm[cl_off(CA_NPHI, j, k, lane, slots, nz)] : lev[LV_NPHI * nz + k];
        double& zs = sm[cl_off(CA_Z, j, k, lane, slots, nz)];
        zz = fma(nk, zz, zs);
        zs = zz;
      }
    }
    {
      const double acc[2] = {accR, accK};
      cl_publish<2>(cluster, acc, busyM, slotM, C);
    }
    cluster.sync();  // every CTA's z and partial sums are in place
    if (threadIdx.x == 0) {
      // ---- the scalar step of Algorithm 1 (as finish_precond_sweep)
      double tot[2];
      cl_totals<2>(slotM, C, tot);
      R = tot[0];
      K = tot[1];
      if (it == 0) R0 = R;
      const double ratio = (R0 > 0.0) ? sqrt(R / R0) : 0.0;
      if (rank == 0) hist[it] = ratio;
      int done = 1;
      if (R0 == 0.0) {
        // r_0 = 0: the initial guess solves the system
      } else if (!(R < INFINITY) || !(R0 < INFINITY)) {
        status = kStBreakdown;
      } else if (ratio < rtol || R == 0.0) {
      } else if (it >= maxit) {
        status = (rtol > 0.0) ? kStNotConv : kStOK;
      } else if (!(K > 0.0)) {
        status = kStBreakdown;
      } else {
        done = 0;
      }
      if (done) {
        iters = it++;
      } else {
        beta = K / kappa_old;
        kappa_old = K;
        ++it;
      }
      sh_done = done;
      sh_beta = beta;
    }
    __syncthreads();
    if (sh_done) break;
    beta = sh_beta;
    // ---- Algorithm 2 sweep on the own tiles (segments of levels per warp),
    // neighbours' z and weights from the owning CTA
    double sig = 0.0;
    for (int unit = warp; unit < slots * segs; unit += kClWarps) {
      const int j = unit % slots, k0 = (unit / slots) * seglen;
      const int k1 = (k0 + seglen < nz) ? k0 + seglen : nz;
      const long long t = (long long)j * C + rank;
      const long long col = t * kTile + lane;
      if (t >= op.ntiles || col >= op.ncols) continue;
      const Nbr nb = neighbours(op, col);
      // owner rank, slot and lane of each horizontal neighbour
      const long long tn[4] = {nb.e >> 5, nb.w >> 5, nb.n >> 5, nb.s >> 5};
      const int ln[4] = {(int)(nb.e & 31), (int)(nb.w & 31), (int)(nb.n & 31), (int)(nb.s & 31)};
      const double* zr[4];
      const double* wr[4];
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        const int own = (int)(tn[d] % C), js = (int)(tn[d] / C);
        const double* base = cluster.map_shared_rank(sm, own);
        zr[d] = base + cl_off(CA_Z, js, 0, ln[d], slots, nz);
        // the west and south weights are the neighbours' east and north ones
        wr[d] = VARY ? base + cl_off(d == 1 ? CA_WE : CA_WN, js, 0, ln[d], slots, nz) : nullptr;
      }
      for (int k = k0; k < k1; ++k) {
        const int kk = k * kTile;
        const double zc = sm[cl_off(CA_Z, j, k, lane, slots, nz)];
        double& us = sm[cl_off(CA_U, j, k, lane, slots, nz)];
        double& ps = sm[cl_off(CA_P, j, k, lane, slots, nz)];
        double& qs = sm[cl_off(CA_Q, j, k, lane, slots, nz)];
        const double pc0 = ps;
        us = fma(alpha, pc0, us);
        const double pc = fma(beta, pc0, zc);
        double a = fma(beta, qs, sm[cl_off(CA_R, j, k, lane, slots, nz)]);
        const double zE = zr[0][kk], zW = zr[1][kk], zN = zr[2][kk], zS = zr[3][kk];
        if (VARY) {
          a = fma(sm[cl_off(CA_WE, j, k, lane, slots, nz)], zE, a);
          a = fma(wr[1][kk], zW, a);
          a = fma(sm[cl_off(CA_WN, j, k, lane, slots, nz)], zN, a);
          a = fma(wr[3][kk], zS, a);
        } else {
          a = fma(lev[LV_HW * nz + k], (zE + zW) + (zN + zS), a);
        }
        sig = fma(pc, a, sig);
        ps = pc;
        qs = a;
      }
    }
    {
      const double acc[1] = {sig};
      cl_publish<1>(cluster, acc, warp < slots * segs, slotA, C);
    }
    cluster.sync();  // every CTA's partial sum is in place; no z is read any more
    if (threadIdx.x == 0) {
      double tot[1];
      cl_totals<1>(slotA, C, tot);
      S = tot[0];
      if (!(S > 0.0) || !(S < INFINITY)) {
        alpha = 0.0;
        iters = it - 1;
        status = kStBreakdown;
        sh_done = 1;
      } else {
        alpha = kappa_old / S;
        sh_done = 0;
      }
      sh_alpha = alpha;
    }
    __syncthreads();
    alpha = sh_alpha;
    if (sh_done) break;
  }
  // ---- u and p back to the row-tiled vectors for the deferred x = u + alpha p
  for (int j = 0; j < slots; ++j) {
    const long long t = (long long)j * C + rank;
    if (t >= op.ntiles) continue;
    for (int e = threadIdx.x; e < nz * kTile; e += kClThreads) {
      const int k = e / kTile, l = e - k * kTile;
      if (t * kTile + l >= op.ncols) continue;
      const long long g = (t * nz + k) * kTile + l;
      u_g[g] = sm[cl_off(CA_U, j, k, l, slots, nz)];
      p_g[g] = sm[cl_off(CA_P, j, k, l, slots, nz)];
    }
  }
  if (rank == 0 && threadIdx.x == 0) {
    st->alpha = alpha;
    st->beta = beta;
    st->kappa_old = kappa_old;
    st->R0 = R0;
    st->last_R = R;
    st->last_kappa = K;
    st->last_sigma = S;
    st->it = it;
    st->iters = iters;
    st->status = status;
    __threadfence();
    st->done = 1;
  }
  cluster.sync();  // no CTA leaves while another may still address its shared memory
}

size_t cl_smem_bytes(const Op& op, int C) {
  const long long slots = (op.ntiles + C - 1) / C;
  return (size_t)(op.varying ? CA_COUNT : CA_U + 1) * slots * op.nz * kTile * sizeof(double);
}

template <bool VARY>
bool cl_launchable(int C, size_t smem) {
  const void* fn = reinterpret_cast<const void*>(k_pcg_cluster<VARY>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      (C > 8 &&
       cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    (void)cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = C;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return n >= 1;
}

}  // namespace

int cluster_ctas(const Op& op) {
  int dev = 0, cl = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, dev) != cudaSuccess || !cl) {
    (void)cudaGetLastError();
    return 0;
  }
  int maxsm = 0;
  cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const size_t room = (size_t)maxsm > 1024 ? (size_t)maxsm - 1024 : 0;  // static slots
  for (int C : {16, 8}) {
    const size_t smem = cl_smem_bytes(op, C);
    if (smem > room) continue;
    const bool ok = op.varying ? cl_launchable<true>(C, smem) : cl_launchable<false>(C, smem);
    if (ok) return C;
  }
  return 0;
}

cudaError_t launch_cluster_loop(const Op& op, DevState* st, double* r, double* u, double* p,
                                double* hist, int C, cudaStream_t s) {
  Op o = op;
  int slots = (int)((op.ntiles + C - 1) / C);
  const size_t smem = cl_smem_bytes(op, C);
  // the dynamic shared memory attribute belongs to the function, not to this
  // context: set it for this launch's size
  const void* fn = op.varying ? reinterpret_cast<const void*>(k_pcg_cluster<true>)
                              : reinterpret_cast<const void*>(k_pcg_cluster<false>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = C;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (op.varying)
    return cudaLaunchKernelEx(&cfg, k_pcg_cluster<true>, o, st, r, u, p, hist, slots);
  return cudaLaunchKernelEx(&cfg, k_pcg_cluster<false>, o, st, r, u, p, hist, slots);
}

}  // namespace pcg
