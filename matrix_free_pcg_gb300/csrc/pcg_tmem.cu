// Column solves of the preconditioner (eq. (19)) with the forward result kept
// in the SM's tensor memory, for the caller's column-contiguous layout.
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs",
// section 4.1 eq. (19) (the Thomas solve per vertical column) and Appendix A
// Algorithm 3 (the fused sweep: r* = r - alpha q, ||r*||^2 and <r*, z>).
//
// Per column the Thomas solve is a forward recurrence whose results w_k are
// consumed in reverse by the back substitution: 8 bytes per cell that must
// live somewhere between the two passes.  Here they live in tensor memory
// (TMEM), the 256 KB per SM that the tensor cores use for accumulators and
// that nothing else on this path needs: each of the 128 TMEM lanes has 512
// 32-bit columns, and a warp reaches the 32 lanes of its sub-partition.  One
// block of 8 warps per SM allocates all 512 columns; warp w uses lanes
// 32(w mod 4) .. 32(w mod 4)+31, one per column of its tile, and columns
// 256 floor(w/4) .. +255, i.e. 128 doubles per grid column (nz <= 128).  The
// w round trip then costs neither L2 traffic nor global load latency, and
// two warps per sub-partition overlap each other's loads and stores with
// their fp64 work (a warp alone adds its operand moves to its fp64 issue).
//
// r (and q) stream through per-warp rings of 8-level chunks in shared
// memory, filled two chunks ahead by 16-byte asynchronous copies in a
// transposed lane mapping (4 lanes per column, 8 columns x 64 contiguous
// bytes per instruction); z leaves through a staging chunk with the same
// coalesced mapping.  The per-cell Thomas factors (row-tiled, one 256-byte
// line per level of a tile) are read straight into registers one chunk
// ahead.
#include <algorithm>

#include "pcg_device.cuh"
#include "pcg_tmem.cuh"

namespace pcg {
namespace {

constexpr int kTwWarps = 8;                  // warps per block: two per sub-partition
constexpr int kTwThreads = kTwWarps * 32;
constexpr int kTwChunk = 8;                  // levels per chunk (ring slot, TMEM region)
constexpr int kTwStages = 3;                 // ring slots per warp
constexpr int kTwCS = kTwChunk + 2;          // ring row (doubles): 80 B, 16-byte aligned
constexpr uint32_t kTwCols = 512;            // TMEM columns of the block: all of the SM's
constexpr uint32_t kTwColsPerWarp = 256;     // per warp: 128 doubles per TMEM lane

// doubles of shared memory per warp: the r (and q) rings and the z staging chunk
template <bool FUSED>
__host__ __device__ constexpr int kTwWarpDoubles() {
  return ((FUSED ? 2 : 1) * kTwStages + 1) * kTile * kTwCS;
}

// Algorithm 3 sweep (FUSED: r* = r - alpha q written back, ||r*||^2 and
// <r*, z> reduced, the scalar step of Algorithm 1 in the last block) or the
// plain solve z = M^{-1} r, on column-contiguous vectors, NZ in {32, 64, 128}.
//
// Warp g of the grid takes tiles g, g + 8G, ... (G blocks), so the
// reductions add in a fixed order.  Per tile: forward y_k = r_k +
// (T_{k-1/2}/D_{k-1}) y_{k-1}, w_k = y_k / D_k into TMEM; backward
// z_k = w_k + (T_{k+1/2}/D_k) z_{k+1}.  <r*, z> is summed in the forward pass
// as sum_k y_k w_k = r*^T L^{-T} D^{-1} L^{-1} r*.
//
// A warp runs the forward pass of its next tile in step with the back
// substitution of its previous one, chunk by chunk (8 levels): two
// independent dependency chains per lane instead of one, so that two warps
// per sub-partition keep the fp64 pipe fed (measured: one chain per warp,
// 0.902 ms, against 0.789 ms on 1024x1024x128).  Both passes share one tile's
// worth of TMEM: step s of the back substitution reads the region that step s
// of the forward pass then overwrites.  For that, the i-th tile of a warp
// keeps its chunk m in region m (i even) or NCH-1-m (i odd): the back
// substitution of tile i-1 consumes its chunks top-down, so at step s both
// passes name the same region.
template <int NZ, bool VARY, bool FUSED>
__global__ void __launch_bounds__(kTwThreads, 1)
    k_precond_tmem(Op op, DevState* st, double* __restrict__ r, const double* __restrict__ q,
                   double* __restrict__ z, double* __restrict__ partials,
                   double* __restrict__ hist) {
  constexpr int C = kTwChunk;
  constexpr int NCH = NZ / C;
  constexpr int FS = VARY ? kTile : 1;  // factor stride between levels
  static_assert(NZ % C == 0, "whole chunks");
  static_assert(2 * NZ <= (int)kTwColsPerWarp, "w of a column fits the warp's TMEM columns");
  extern __shared__ __align__(16) double smem[];
  __shared__ uint32_t tmem_base_s;
  if (FUSED && ld_done(st)) return;  // set by an earlier launch: the same in every thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, kTwCols);
    tmem_relinquish();
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  // this warp's TMEM: lane field 32 (w mod 4), its half of the columns
  const uint32_t tw = tmem_base_s + ((uint32_t)(32 * (warp & 3)) << 16) +
                      kTwColsPerWarp * (uint32_t)(warp >> 2);
  double* Rg = smem + (size_t)warp * kTwWarpDoubles<FUSED>();  // [kTwStages][32][kTwCS]
  double* Qg = Rg + kTwStages * kTile * kTwCS;                  // FUSED only
  double* Zs = Rg + (FUSED ? 2 : 1) * kTwStages * kTile * kTwCS;  // [32][kTwCS]
  const double nalpha = FUSED ? -st->alpha : 0.0;
  // copy mapping: 4 lanes x 16 bytes per column chunk, 8 columns per instruction
  const int cq = lane >> 2, pp = 2 * (lane & 3);
  const uint64_t keep = l2_keep(), stream = l2_stream();
  double accR0 = 0.0, accR1 = 0.0, accK0 = 0.0, accK1 = 0.0;
  auto ldf = [&](const double* a, uint64_t pol) { return VARY ? ld_hint(a, pol) : __ldg(a); };
  const long long G = (long long)gridDim.x * kTwWarps;
  const long long tfirst = (long long)blockIdx.x * kTwWarps + warp;
  auto ncols_of = [&](long long t) { return (int)min((long long)kTile, op.ncols - t * kTile); };
  auto fi_of = [&](long long t) {
    return VARY ? op.tinvd + t * NZ * kTile + lane : op.lev + LV_INVD * NZ;
  };
  auto fn_of = [&](long long t) {
    return VARY ? op.tnphi + t * NZ * kTile + lane : op.lev + LV_NPHI * NZ;
  };
  auto region = [&](long long i, int m) { return (i & 1) ? NCH - 1 - m : m; };
  // Forward positions p = i*NCH + m (chunk m of the warp's i-th tile) stream
  // through the ring: slot p mod kTwStages, copied kTwStages-1 positions ahead,
  // one commit group per position (empty past the warp's last tile).
  auto issue_pos = [&](long long p) {
    const long long t = tfirst + (p / NCH) * G;
    if (t < op.ntiles) {
      const int m = (int)(p % NCH), sl = (int)(p % kTwStages), nc = ncols_of(t);
      const long long col0 = t * kTile;
#pragma unroll
      for (int i = 0; i < kTile / 8; ++i) {
        const int c = cq + 8 * i;
        if (c < nc) {
          const long long g = (col0 + c) * NZ + m * C + pp;
          cp_async16_hint(Rg + (sl * kTile + c) * kTwCS + pp, r + g, stream);
          if (FUSED) cp_async16_hint(Qg + (sl * kTile + c) * kTwCS + pp, q + g, stream);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int p = 0; p < kTwStages - 1; ++p) issue_pos(p);

  // forward state (tile tf = the warp's i-th tile) and backward state (tile tb)
  double y = 0.0, nprev = 0.0, zz = 0.0;
  double ci[C] = {}, cn[C] = {}, ni[C] = {}, nn[C] = {}, ww[C] = {}, bw[C] = {}, bn[C] = {},
         nb[C] = {};
  // one forward chunk m of tile tf (position p), with the factors of the next
  // chunk (or of the next tile's first) fetched meanwhile
  auto fwd_begin = [&](long long p) {
    issue_pos(p + kTwStages - 1);
    cp_async_wait<kTwStages - 1>();  // position p has landed (this lane's copies)
    __syncwarp();                    // ... and everyone else's
  };
  auto fwd_level = [&](int sl, int j, int nc) {
    const double* rs = Rg + (sl * kTile + lane) * kTwCS;
    const double* qs = Qg + (sl * kTile + lane) * kTwCS;
    if (lane < nc) {
      const double2 rv = lds2(rs + j);
      double r0 = rv.x, r1 = rv.y;
      if (FUSED) {
        const double2 qv = lds2(qs + j);
        r0 = fma(nalpha, qv.x, r0);
        r1 = fma(nalpha, qv.y, r1);
        accR0 = fma(r0, r0, accR0);
        accR1 = fma(r1, r1, accR1);
        sts2(Rg + (sl * kTile + lane) * kTwCS + j, r0, r1);
      }
      y = fma(nprev, y, r0);
      ww[j] = y * ci[j];
      if (FUSED) accK0 = fma(y, ww[j], accK0);
      y = fma(cn[j], y, r1);
      ww[j + 1] = y * ci[j + 1];
      if (FUSED) accK1 = fma(y, ww[j + 1], accK1);
      nprev = cn[j + 1];
    }
  };
  auto bwd_pair = [&](int c, int j, int nc) {  // levels c*C+j and c*C+j-1 (j odd)
    if (lane < nc) {
      const int k = c * C + j;
      const double zh = (k == NZ - 1) ? bw[j] : fma(bn[j], zz, bw[j]);
      zz = fma(bn[j - 1], zh, bw[j - 1]);
      sts2(Zs + lane * kTwCS + j - 1, zz, zh);
    }
  };
  auto fwd_end = [&](long long t, int m, int sl, int nc) {  // r* of the chunk back out
    if (FUSED) {
      __syncwarp();
      const long long col0 = t * kTile;
#pragma unroll
      for (int i = 0; i < kTile / 8; ++i) {
        const int c = cq + 8 * i;
        if (c < nc)
          st2_hint(r + (col0 + c) * NZ + m * C + pp, lds2(Rg + (sl * kTile + c) * kTwCS + pp),
                   stream);
      }
    }
  };
  auto bwd_end = [&](long long t, int c, int nc) {  // z of the chunk out, transposed
    __syncwarp();
    const long long col0 = t * kTile;
#pragma unroll
    for (int i = 0; i < kTile / 8; ++i) {
      const int cc = cq + 8 * i;
      if (cc < nc) st2_hint(z + (col0 + cc) * NZ + c * C + pp, lds2(Zs + cc * kTwCS + pp), stream);
    }
  };
  auto load_fwd_factors = [&](long long t, int m, double (&a)[C], double (&b)[C]) {
    const double* fi = fi_of(t);
    const double* fn = fn_of(t);
#pragma unroll
    for (int j = 0; j < C; ++j) {
      a[j] = ldf(fi + (m * C + j) * FS, stream);
      b[j] = ldf(fn + (m * C + j) * FS, keep);
    }
  };
  auto load_bwd_factors = [&](long long t, int c, double (&b)[C]) {
    const double* fn = fn_of(t);
#pragma unroll
    for (int j = 0; j < C; ++j) b[j] = ldf(fn + (c * C + j) * FS, stream);
  };

  long long i = 0;  // the warp's tile index: tf = tfirst + i*G
  if (tfirst < op.ntiles) {
    // ---- first tile: forward pass alone
    const long long tf = tfirst;
    const int ncf = ncols_of(tf);
    load_fwd_factors(tf, 0, ci, cn);
#pragma unroll 1
    for (int m = 0; m < NCH; ++m) {
      const long long p = m;
      const int sl = (int)(p % kTwStages);
      if (m + 1 < NCH) load_fwd_factors(tf, m + 1, ni, nn);
      fwd_begin(p);
#pragma unroll
      for (int j = 0; j < C; j += 2) fwd_level(sl, j, ncf);
      tmem_st8(tw + 2u * C * (uint32_t)region(0, m), ww);
      fwd_end(tf, m, sl, ncf);
      __syncwarp();
      if (m + 1 < NCH) {
#pragma unroll
        for (int j = 0; j < C; ++j) {
          ci[j] = ni[j];
          cn[j] = nn[j];
        }
      }
    }
    tmem_wait_st();
    // ---- steady state: tile i's forward pass in step with tile i-1's back
    // substitution; then the last tile's back substitution alone
#pragma unroll 1
    for (i = 1;; ++i) {
      const long long tb = tfirst + (i - 1) * G, tf2 = tb + G;
      const bool fwd = tf2 < op.ntiles;
      const int ncb = ncols_of(tb), ncf2 = fwd ? ncols_of(tf2) : 0;
      y = 0.0;
      nprev = 0.0;
      zz = 0.0;
      load_bwd_factors(tb, NCH - 1, bn);
      if (fwd) load_fwd_factors(tf2, 0, ci, cn);
#pragma unroll 1
      for (int s = 0; s < NCH; ++s) {
        const int c = NCH - 1 - s;  // the back substitution's chunk
        const int rg = region(i - 1, c);
        if (c > 0) load_bwd_factors(tb, c - 1, nb);
        if (fwd && s + 1 < NCH) load_fwd_factors(tf2, s + 1, ni, nn);
        tmem_ld8(tw + 2u * C * (uint32_t)rg, bw);  // complete on return
        const long long p = i * NCH + s;
        const int sl = (int)(p % kTwStages);
        if (fwd) fwd_begin(p);
        // the two passes' levels interleaved: independent chains
#pragma unroll
        for (int j = 0; j < C; j += 2) {
          if (fwd) fwd_level(sl, j, ncf2);
          bwd_pair(c, C - 1 - j, ncb);
        }
        if (fwd) {
          tmem_st8(tw + 2u * C * (uint32_t)rg, ww);  // the region just read: region(i, s)
          fwd_end(tf2, s, sl, ncf2);
        }
        bwd_end(tb, c, ncb);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < C; ++j) bn[j] = nb[j];
        if (fwd && s + 1 < NCH) {
#pragma unroll
          for (int j = 0; j < C; ++j) {
            ci[j] = ni[j];
            cn[j] = nn[j];
          }
        }
      }
      if (!fwd) break;
      tmem_wait_st();
    }
  }
  cp_async_wait<0>();
  // every warp is done with TMEM before warp 0 frees it
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem_base_s, kTwCols);
  if (FUSED) {
    double R, K;
    if (grid_sum2<kTwThreads>(accR0 + accR1, accK0 + accK1, partials, &st->ticket_m, R, K))
      finish_precond_sweep(st, R, K, hist);
  }
}

template <int NZ, bool VARY, bool FUSED>
cudaError_t launch_nz(const Op& op, DevState* st, double* r, const double* q, double* z,
                      double* partials, double* hist, int grid, size_t smem, cudaStream_t s) {
  k_precond_tmem<NZ, VARY, FUSED><<<grid, kTwThreads, smem, s>>>(op, st, r, q, z, partials, hist);
  return cudaGetLastError();
}

template <bool VARY, bool FUSED>
cudaError_t launch_vary(const Op& op, DevState* st, double* r, const double* q, double* z,
                        double* partials, double* hist, int grid, size_t smem, cudaStream_t s) {
  switch (op.nz) {
    case 128:
      return launch_nz<128, VARY, FUSED>(op, st, r, q, z, partials, hist, grid, smem, s);
    case 64:
      return launch_nz<64, VARY, FUSED>(op, st, r, q, z, partials, hist, grid, smem, s);
    default:
      return launch_nz<32, VARY, FUSED>(op, st, r, q, z, partials, hist, grid, smem, s);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Dynamic shared memory of a launch: the rings of its 8 warps, padded past
// half of the SM's shared memory so that no second block -- which would wait
// in tcgen05.alloc for the first one's columns -- is placed on the SM.
int tmem_smem_bytes(bool fused) {
  int dev = 0, smem_sm = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int need = (int)sizeof(double) * kTwWarps *
                   (fused ? kTwWarpDoubles<true>() : kTwWarpDoubles<false>());
  const int pad = smem_sm / 2 + 1024;
  return std::min(std::max(need, pad), optin - 1024);
}

}  // namespace

bool precond_tmem_supported(const Op& op, const double* r, const double* q, const double* z) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (op.nz == 32 || op.nz == 64 || op.nz == 128) && al16(r) && al16(z) && (!q || al16(q));
}

cudaError_t prepare_precond_tmem() {
  const int b0 = tmem_smem_bytes(false), b1 = tmem_smem_bytes(true);
  cudaError_t e = cudaSuccess, x;
#define PCG_TW_SET(NZ, V)                                                   \
  if ((x = set_smem(k_precond_tmem<NZ, V, false>, b0)) != cudaSuccess) e = x; \
  if ((x = set_smem(k_precond_tmem<NZ, V, true>, b1)) != cudaSuccess) e = x;
  PCG_TW_SET(128, true) PCG_TW_SET(128, false) PCG_TW_SET(64, true) PCG_TW_SET(64, false)
  PCG_TW_SET(32, true) PCG_TW_SET(32, false)
#undef PCG_TW_SET
  return e;
}

int grid_precond_tmem(const Op& op, int num_sms) {
  const long long work = (op.ntiles + kTwWarps - 1) / kTwWarps;  // blocks that get a tile
  return (int)std::max(1LL, std::min((long long)num_sms, work));
}


cudaError_t launch_precond_tmem(const Op& op, DevState* st, double* r, const double* q, double* z,
                                double* partials, double* hist, bool fused, int grid,
                                cudaStream_t s) {
  const size_t smem = (size_t)tmem_smem_bytes(fused);
  if (fused)
    return op.varying ? launch_vary<true, true>(op, st, r, q, z, partials, hist, grid, smem, s)
                      : launch_vary<false, true>(op, st, r, q, z, partials, hist, grid, smem, s);
  return op.varying ? launch_vary<true, false>(op, st, r, q, z, partials, hist, grid, smem, s)
                    : launch_vary<false, false>(op, st, r, q, z, partials, hist, grid, smem, s);
}

}  // namespace pcg
