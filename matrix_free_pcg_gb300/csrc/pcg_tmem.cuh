// Tensor-memory (TMEM) wrappers of the column-layout kernels that keep the
// Thomas forward pass's w in the SM's tensor memory (pcg_tmem.cu; the
// row-tiled sweep keeps w in L2 instead).  TMEM is the 256 KB
// per SM that the tensor cores use for accumulators: 128 lanes of 512 32-bit
// columns; a warp reaches the 32 lanes of its sub-partition (warp w of a
// block: lanes 32 (w mod 4) .. +31).  Internal; internal linkage.
#pragma once

#include <cstdint>

#include "pcg_device.cuh"

namespace pcg {
namespace {

// ---- tensor memory (tcgen05) wrappers; every one is warp-wide (.sync.aligned)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 8 doubles of this thread into 16 consecutive columns of its TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const double (&v)[8]) {
  uint32_t u[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    u[2 * j] = (uint32_t)__double2loint(v[j]);
    u[2 * j + 1] = (uint32_t)__double2hiint(v[j]);
  }
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
      "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]),
      "r"(u[15])
      : "memory");
}

// The 8 doubles stored by tmem_st8 at taddr, back into this thread's
// registers; the load is complete (tcgen05.wait::ld) when this returns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, double (&v)[8]) {
  uint32_t u[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
        "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
        "=r"(u[14]), "=r"(u[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __hiloint2double((int)u[2 * j + 1], (int)u[2 * j]);
}

}  // namespace
}  // namespace pcg
