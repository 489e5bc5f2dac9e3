// Preconditioner solve with its inner product, for callers that cannot
// allocate device memory when they call.
//
// pcg_precond_dot_noalloc (include/pcg.h) computes z = M^{-1} r and
// <r, z> like the preconditioner sweep does, but takes its scratch memory --
// one partial sum per 32-column tile -- from a fixed array compiled into
// this library instead of from an allocation.  Some callers must not call
// cudaMalloc/cudaFree while they run: code that must not synchronise the
// device (cudaFree does, and cudaMalloc may), or applications that reserve
// all device memory for their own pool at start-up.  The operator tables
// still come from a context made beforehand with pcg_create.
//
// The scratch array lives in every GPU that loads this library until the
// process exits.  In host code its name is only a stand-in for the device
// copy, so pcg_create looks up the real device address with
// cudaGetSymbolAddress (with the context's device current) and keeps it in
// the context; that lookup also loads this file's module on the device, so
// the entry point itself neither loads code nor allocates.
#include <cstdint>

#include "pcg_internal.h"

namespace pcg {
namespace {

// Scratch: one partial sum of <r, z> per tile of 32 columns.  Every call
// writes the partial of every tile of its grid before reading any of them,
// so nothing has to be cleared between calls.  Calls that overlap on the GPU
// (two streams, two host threads) race on this array.
static __device__ __align__(256) double g_tile_partials[kNoallocMaxTiles];

// One warp per tile of 32 columns, one column per lane, walking its column
// in global memory: forward y_k = r_k + (T_{k-1/2}/D_{k-1}) y_{k-1} with
// w_k = y_k / D_k written into z, then back substitution
// z_k = w_k + (T_{k+1/2}/D_k) z_{k+1} and the partial sum of r_k z_k.
__global__ void k_precond_dot_tiles(Op op, const double* __restrict__ r,
                                    double* __restrict__ z, double* __restrict__ partials) {
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int nz = op.nz;
  for (long long t = warp; t < op.ntiles; t += nwarps) {
    const long long col = t * kTile + lane;
    double acc = 0.0;
    if (col < op.ncols) {
      const double* rc = r + col * nz;
      double* zc = z + col * nz;
      const double* fn = op.varying ? op.tnphi + t * nz * kTile + lane : op.lev + LV_NPHI * nz;
      const double* fi = op.varying ? op.tinvd + t * nz * kTile + lane : op.lev + LV_INVD * nz;
      const int fs = op.varying ? kTile : 1;
      double y = 0.0, nprev = 0.0;
      for (int k = 0; k < nz; ++k) {
        y = fma(nprev, y, rc[k]);
        zc[k] = y * fi[k * fs];
        nprev = fn[k * fs];
      }
      double zz = zc[nz - 1];
      acc = fma(rc[nz - 1], zz, acc);
      for (int k = nz - 2; k >= 0; --k) {
        zz = fma(fn[k * fs], zz, zc[k]);
        zc[k] = zz;
        acc = fma(rc[k], zz, acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
    if (lane == 0) partials[t] = acc;
  }
}

// Sum of the tile partials in a fixed order (the same result on every call).
__global__ void k_sum_tiles(const double* __restrict__ partials, long long ntiles,
                            double* __restrict__ out) {
  __shared__ double sh[256];
  double a = 0.0;
  for (long long i = threadIdx.x; i < ntiles; i += blockDim.x) a += partials[i];
  sh[threadIdx.x] = a;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = sh[0];
}

}  // namespace

cudaError_t noalloc_scratch_address(double** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_tile_partials);
  if (e == cudaSuccess) *out = static_cast<double*>(p);
  return e;
}

cudaError_t launch_precond_dot_noalloc(const Op& op, const double* r, double* z, double* rz,
                                       double* partials, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  long long blocks = (op.ntiles + 7) / 8;  // 8 warps (tiles) per block of 256 threads
  const long long cap = 8LL * num_sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  k_precond_dot_tiles<<<(int)blocks, 256, 0, s>>>(op, r, z, partials);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_sum_tiles<<<1, 256, 0, s>>>(partials, op.ntiles, rz);
  return cudaGetLastError();
}

}  // namespace pcg
