// Device-side helpers shared by the kernel files of the solver: vector
// loads and stores, the periodic neighbour map, the deterministic grid
// reduction with the scalar step of Algorithm 1 that follows the
// preconditioner sweep (Mueller, Guo, Scheichl, Shi, "Matrix-free GPU
// implementation of a preconditioned conjugate gradient solver for
// anisotropic elliptic PDEs", section 4.3 and Appendix A), and the cp.async /
// L2 cache-hint wrappers.  Internal; every definition has internal linkage.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pcg_internal.h"

namespace pcg {
namespace {

constexpr int kStOK = 0, kStNotConv = 4, kStBreakdown = 5, kStTimeout = 6;

__device__ __forceinline__ double2 ld2(const double* p) {
  return *reinterpret_cast<const double2*>(p);
}
__device__ __forceinline__ double2 ldg2(const double* p) {
  return __ldg(reinterpret_cast<const double2*>(p));
}
__device__ __forceinline__ void st2(double* p, double2 v) {
  *reinterpret_cast<double2*>(p) = v;
}
__device__ __forceinline__ int ld_done(const DevState* st) {
  return *reinterpret_cast<const volatile int*>(&st->done);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Horizontal neighbours of a column, periodic in i and j.
struct Nbr {
  long long e, w, n, s;
};
__device__ __forceinline__ Nbr neighbours(const Op& op, long long col) {
  const long long j = col / op.nx;
  const int i = (int)(col - j * op.nx);
  Nbr nb;
  nb.e = (i == op.nx - 1) ? col - (op.nx - 1) : col + 1;
  nb.w = (i == 0) ? col + (op.nx - 1) : col - 1;
  nb.n = (j == op.ny - 1) ? col - (long long)(op.ny - 1) * op.nx : col + op.nx;
  nb.s = (j == 0) ? col + (long long)(op.ny - 1) * op.nx : col - op.nx;
  return nb;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Deterministic grid reduction of two values: warp shuffle tree -> block
// (fixed order) -> per-block partials -> the last block to take a ticket sums
// the partials in block order.  No block ever waits on another.  Returns true
// in thread 0 of the last block, with the totals in tot0/tot1.
template <int NT>
__device__ bool grid_sum2(double v0, double v1, double* __restrict__ partials,
                          unsigned int* ticket, double& tot0, double& tot1) {
  constexpr int NW = NT / 32;
  __shared__ double sh0[NW], sh1[NW];
  __shared__ bool am_last;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v0 = warp_sum(v0);
  v1 = warp_sum(v1);
  if (NW > 1) {
    if (lane == 0) {
      sh0[w] = v0;
      sh1[w] = v1;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double a = v0, b = v1;
    for (int i = 1; i < NW; ++i) {
      a += sh0[i];
      b += sh1[i];
    }
    partials[2 * blockIdx.x] = a;
    partials[2 * blockIdx.x + 1] = b;
    __threadfence();
    const unsigned int t = atomicAdd(ticket, 1u);
    am_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!am_last) return false;
  __threadfence();
  double a = 0.0, b = 0.0;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += NT) {
    a += __ldcg(partials + 2 * i);
    b += __ldcg(partials + 2 * i + 1);
  }
  a = warp_sum(a);
  b = warp_sum(b);
  if (NW > 1) {
    if (lane == 0) {
      sh0[w] = a;
      sh1[w] = b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int i = 1; i < NW; ++i) {
      a += sh0[i];
      b += sh1[i];
    }
    tot0 = a;
    tot1 = b;
    *ticket = 0u;
  }
  return threadIdx.x == 0;
}

// Last-block bookkeeping of Algorithm 1 after the preconditioner sweep of
// iteration it: ||r||, stopping test, beta = kappa/kappa_old.
__device__ void finish_precond_sweep(DevState* st, double R, double K, double* hist) {
  const int it = st->it;
  if (it == 0) st->R0 = R;
  const double R0 = st->R0;
  st->last_R = R;
  st->last_kappa = K;
  const double ratio = (R0 > 0.0) ? sqrt(R / R0) : 0.0;
  hist[it] = ratio;
  int done = 0, status = kStOK;
  if (st->dev_error) {
    done = 1;
    status = kStTimeout;
  } else if (R0 == 0.0) {
    done = 1;  // r_0 = 0: the initial guess solves the system
  } else if (!(R < INFINITY) || !(R0 < INFINITY)) {
    done = 1;
    status = kStBreakdown;  // NaN or Inf in the residual
  } else if (ratio < st->rtol || R == 0.0) {
    done = 1;
  } else if (it >= st->maxit) {
    done = 1;
    status = (st->rtol > 0.0) ? kStNotConv : kStOK;
  } else if (!(K > 0.0)) {
    done = 1;
    status = kStBreakdown;
  } else {
    st->beta = K / st->kappa_old;
    st->kappa_old = K;
  }
  if (done) {
    st->iters = it;
    st->status = status;
    __threadfence();
    st->done = 1;
  }
  st->it = it + 1;
}

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// L2 eviction-priority hints: data read again soon (the w scratch, the
// Thomas factors the backward sweep reads a second time) is kept, data that
// streams through once is let go first.
__device__ __forceinline__ uint64_t l2_keep() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_stream() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async16_hint(void* dst_smem, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_hint(double* a, double v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f64 [%0], %1, %2;" ::"l"(a), "d"(v), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st2_hint(double* a, double2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f64 [%0], {%1, %2}, %3;" ::"l"(a), "d"(v.x),
               "d"(v.y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ double ld_hint(const double* a, uint64_t pol) {
  double v;
  asm volatile("ld.global.L2::cache_hint.f64 %0, [%1], %2;" : "=d"(v) : "l"(a), "l"(pol)
               : "memory");
  return v;
}

// Grid-wide barrier for a cooperative launch (every block resident), on a
// counter that only grows during the launch (zeroed before it).  Thread 0 of
// each block publishes the block's writes, adds its arrival (a reduction in
// L2: no value comes back) and polls until the count reaches `target` =
// nblocks times the number of barriers passed so far, this one included.
// Nothing is reset or released after the last arrival: a waiting block sees
// the barrier open on its next poll.  The poll gives up after `wait_ns`
// nanoseconds of the global timer, or after `limit` tries, whichever comes
// first; the block then records the timeout in *err and the barrier returns false
// (the caller leaves its loop; nothing waits without bound).  Global writes
// made before the barrier are visible to every block after it (read them
// with __ldcg, past the non-coherent L1).  The unsigned difference keeps the
// test right across a wrap of the counter.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool grid_barrier(unsigned int* count, unsigned int target, int* err,
                                             long long limit, unsigned long long wait_ns) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(count, 1u);
    const unsigned long long t0 = global_ns();
    long long polls = 0;
    while ((int)(*reinterpret_cast<volatile unsigned int*>(count) - target) < 0) {
      if (++polls > limit || global_ns() - t0 > wait_ns) {
        ok = 0;
        atomicExch(err, 1);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

__device__ __forceinline__ double2 lds2(const double* p) {
  return *reinterpret_cast<const double2*>(p);
}
__device__ __forceinline__ void sts2(double* p, double a, double b) {
  *reinterpret_cast<double2*>(p) = make_double2(a, b);
}

}  // namespace
}  // namespace pcg
