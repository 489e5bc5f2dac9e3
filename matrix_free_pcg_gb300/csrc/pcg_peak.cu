// Measured fp64 rate of the device's non-tensor pipe: the denominator of the
// roofline of the two sweeps, whose work is fp64 fused multiply-adds, products
// and sums with no dense contraction (the paper reports measured per-kernel
// rates, section 7 Table 7; this gives the rate the GPU itself can reach).
//
// Each thread carries kChains independent chains a <- a*m + c of fp64 fused
// multiply-adds, so that no instruction waits on its predecessor and the only
// limit is how fast the pipe retires them.  Thread 0 of every block reads
// clock64() and the global nanosecond timer at its start and end: their
// ratio is the SM clock during the launch.
#include "pcg_internal.h"

namespace pcg {
namespace {

constexpr int kChains = 8;   // independent chains per thread
constexpr int kUnroll = 16;  // FMAs per chain per loop trip

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void k_fp64_fma_rate(int trips, double m, double c, double* __restrict__ sink,
                                unsigned long long* __restrict__ stamps) {
  unsigned long long c0 = 0, t0 = 0;
  if (threadIdx.x == 0) {
    t0 = global_ns();
    c0 = clock64();
  }
  double a[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) a[j] = c * (double)(threadIdx.x + 1 + j);
  for (int t = 0; t < trips; ++t) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
      for (int j = 0; j < kChains; ++j) a[j] = fma(a[j], m, c);
    }
  }
  double s = 0.0;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += a[j];
  // the chains converge to c/(1-m) > 0: this store never happens, but the
  // compiler cannot know it and has to compute every chain
  if (s < 0.0) sink[blockIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long c1 = clock64(), t1 = global_ns();
    stamps[2 * blockIdx.x] = c1 - c0;
    stamps[2 * blockIdx.x + 1] = t1 - t0;
  }
}

}  // namespace

long long fp64_rate_lane_ops(int blocks, int threads, int trips) {
  return (long long)blocks * threads * trips * kUnroll * kChains;
}

cudaError_t launch_fp64_rate(int blocks, int threads, int trips, double* sink,
                             unsigned long long* stamps, cudaStream_t s) {
  // m < 1 and c > 0 keep every chain positive and bounded, away from
  // subnormals and overflow
  k_fp64_fma_rate<<<blocks, threads, 0, s>>>(trips, 1.0 - 1.0 / 1024.0, 1.0 / 4096.0, sink,
                                             stamps);
  return cudaGetLastError();
}

}  // namespace pcg
