// Coefficient set-up kernels of the matrix-free PCG solver (fp64, sm_103a).
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs":
// the face values and the diagonal of the operator, section 3 eqs. (5)-(8)
// and section 4.2 eq. (18); the Thomas factors of the column blocks of the
// preconditioner, section 4.1 eq. (19).  Run once per operator (pcg_create,
// pcg_update_coeffs).
#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "pcg_device.cuh"
#include "pcg_internal.h"

namespace pcg {
namespace {

__global__ void k_face_coeffs(Op op, double* __restrict__ faceE, double* __restrict__ faceN) {
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < op.ncols;
       c += (long long)gridDim.x * blockDim.x) {
    const Nbr nb = neighbours(op, c);
    faceE[c] = 0.5 * (op.ah[c] + op.ah[nb.e]);
    faceN[c] = 0.5 * (op.ah[c] + op.ah[nb.n]);
  }
}

// The admissibility check of an uploaded a_h field (finite and >= 0, as the
// operator of eqs. (5)-(8) needs), on its staging copy: every offending
// thread stores the same 1.
__global__ void k_check_field(const double* __restrict__ f, long long n, int* err) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const double v = f[i];
    if (!(v >= 0.0 && v <= DBL_MAX)) *err = 1;
  }
}

// T/D rounded to nearest, from y = 1/D rounded to nearest, by Markstein's
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990; Markstein's
// theorem in Muller et al., "Handbook of Floating-Point Arithmetic"): with
// y within half an ulp of 1/D and q within one ulp of T/D, the remainder
// T - D q is exact as a fused multiply-add and q + (T - D q) y rounds to
// T/D.  The first correction makes q = RN(T y) faithful, the second rounds
// it.  Valid for the positive, normal operands of the Thomas set-up; bitwise
// equal to the IEEE quotient (the row-tiled sweep that rebuilds its factors
// divides, and the tests compare the two).
__device__ __forceinline__ double quotient_rn(double T, double D, double y) {
  double q = T * y;
  double r = fma(-q, D, T);
  q = fma(r, y, q);
  r = fma(-q, D, T);
  return fma(r, y, q);
}

// Per-cell tables of an a_h field, one thread per column (eqs. (8), (18),
// (19)): the diagonal h_k*mass + T_{k+1/2} + T_{k-1/2} + h_k * (sum of the
// four face values), stored column-contiguously and, when the context holds
// the row-tiled copy, row-tiled; the horizontal weights -h_k a_E and -h_k a_N
// of the row-tiled stencil sweep; and the Thomas factors of the column in the
// LDL^T form used by the sweeps, D_k = diag_k - T_{k-1/2} (T_{k-1/2}/D_{k-1}),
// stored as T_{k+1/2}/D_k and 1/D_k, row-tiled, so that a warp reads 32
// columns' level k as one 256-byte line.
//
// The diagonal and the pivots are formed with explicitly rounded operations
// (no fused multiply-add): the column systems of strongly graded, strongly
// anisotropic grids amplify a one-ulp change of a pivot by up to ~1e5 in the
// solution, so they are formed exactly as their definition rounds them
// (product rounded, then sum), the numbers any plain fp64 evaluation of
// eq. (19) produces.  1/D_k is the IEEE reciprocal; T_{k+1/2}/D_k is derived
// from it exactly (quotient_rn).
__global__ void k_column_setup(Op op, DevState* st, double* __restrict__ cdiag,
                               double* __restrict__ cdiag_t, double* __restrict__ cwE_t,
                               double* __restrict__ cwN_t, double* __restrict__ tnphi,
                               double* __restrict__ tinvd) {
  const int nz = op.nz;
  const double* __restrict__ lev = op.lev;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < op.ncols;
       c += (long long)gridDim.x * blockDim.x) {
    const long long t = c / kTile;
    const int lane = (int)(c - t * kTile);
    const Nbr nb = neighbours(op, c);
    const double sf = op.faceE[c] + op.faceE[nb.w] + op.faceN[c] + op.faceN[nb.s];
    double nphi_prev = 0.0;
    int bad = 0;
    for (int k = 0; k < nz; ++k) {
      const double diag = __dadd_rn(lev[LV_DIAG * nz + k], __dmul_rn(lev[LV_H * nz + k], sf));
      const long long o = (t * nz + k) * kTile + lane;
      cdiag[c * nz + k] = diag;
      if (cdiag_t) cdiag_t[o] = diag;
      if (cwE_t) {  // horizontal weights -h_k a_f of the east and north faces
        cwE_t[o] = __dmul_rn(lev[LV_HW * nz + k], op.faceE[c]);
        cwN_t[o] = __dmul_rn(lev[LV_HW * nz + k], op.faceN[c]);
      }
      const double D = __dsub_rn(diag, __dmul_rn(lev[LV_TDN * nz + k], nphi_prev));
      if (!(D > 0.0)) bad = 1;
      const double invd = __drcp_rn(D);  // 1/D rounded to nearest
      const double nphi = quotient_rn(lev[LV_TUP * nz + k], D, invd);
      tnphi[o] = nphi;
      tinvd[o] = invd;
      nphi_prev = nphi;
    }
    if (bad) st->setup_error = 1;
  }
}

}  // namespace

cudaError_t launch_face_coeffs(const Op& op, double* faceE, double* faceN, cudaStream_t s) {
  long long g = (op.ncols + 255) / 256;
  if (g > 65536) g = 65536;
  k_face_coeffs<<<(int)g, 256, 0, s>>>(op, faceE, faceN);
  return cudaGetLastError();
}

__global__ void k_flag_to_host(const int* src, int* dst) { *dst = *src; }

cudaError_t launch_flag_to_host(const int* src, int* dst, cudaStream_t s) {
  k_flag_to_host<<<1, 1, 0, s>>>(src, dst);
  return cudaGetLastError();
}

cudaError_t launch_check_field(const double* f, long long n, int* err, cudaStream_t s) {
  long long g = (n + 255) / 256;
  if (g > 4096) g = 4096;
  k_check_field<<<(int)std::max<long long>(g, 1), 256, 0, s>>>(f, n, err);
  return cudaGetLastError();
}

cudaError_t launch_column_setup(const Op& op, DevState* st, double* cdiag, double* cdiag_t,
                                double* cwE_t, double* cwN_t, double* tnphi, double* tinvd,
                                cudaStream_t s) {
  long long g = (op.ncols + 127) / 128;
  if (g > 65536) g = 65536;
  k_column_setup<<<(int)g, 128, 0, s>>>(op, st, cdiag, cdiag_t, cwE_t, cwN_t, tnphi, tinvd);
  return cudaGetLastError();
}

}  // namespace pcg
