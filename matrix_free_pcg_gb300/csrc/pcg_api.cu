// Host driver and C ABI of libpcg (declared in include/pcg.h).
//
// Method: Mueller, Guo, Scheichl, Shi, "Matrix-free GPU implementation of a
// preconditioned conjugate gradient solver for anisotropic elliptic PDEs":
// the interleaved PCG loop of section 4.3, Algorithm 1, driven from the host
// with all data and all scalars resident on the device (section 6: only the
// initial solution and right-hand side go in, the solution comes out).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <cfloat>
#include <functional>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/pcg.h"
#include "pcg_internal.h"

using pcg::DevState;
using pcg::Op;

namespace {

thread_local std::string g_create_error = "no error";

struct KernelEvent {
  int kind;
  cudaEvent_t start, stop;
};

// One batch of the row-tiled solve loop (preconditioner and stencil sweeps of
// `iters` iterations) as an instantiated CUDA graph.  With timing, event-record
// nodes mark the boundaries between consecutive kernels: ev[2i] before the
// preconditioner sweep of iteration i, ev[2i+1] between it and the stencil
// sweep, ev[2i+2] after that (2*iters+1 events; each costs GPU time, so
// neighbours share one).
struct BatchGraph {
  cudaGraphExec_t exec = nullptr;
  std::vector<cudaEvent_t> ev;
};

}  // namespace

struct pcg_ctx {
  int device = -1;
  int num_sms = 0;
  cudaStream_t stream = nullptr;
  Op op{};
  bool has_field_buffers = false;
  // device buffers owned by the context
  double *r = nullptr, *z = nullptr, *p = nullptr, *q = nullptr;
  double *lev = nullptr, *ah = nullptr, *faceE = nullptr, *faceN = nullptr;
  double* ah_stage = nullptr;  // an uploaded a_h field, checked here before it replaces ah
  double *cdiag = nullptr, *tnphi = nullptr, *tinvd = nullptr;
  double *partials = nullptr, *hist = nullptr, *wscratch = nullptr;
  int layout = PCG_LAYOUT_COLUMN;       // layout of the solver's internal vectors
  double *u_t = nullptr, *cdiag_t = nullptr;  // row-tiled layout: iterate, diagonal
  double *cwE_t = nullptr, *cwN_t = nullptr;  // row-tiled layout: horizontal weights
  int grid_tm = 1, grid_ta = 1;  // row-tiled preconditioner / stencil sweeps
  int factors = PCG_FACTORS_STORED;  // per-cell factors read (stored) or rebuilt per sweep
  double* nscratch = nullptr;        // recompute: per-warp T_{k+1/2}/D_k scratch
  // substructured column solve: requested blocks (0 automatic), blocks in use, grid
  int split_req = 0, split_p = 1, grid_sp = 0;
  int loop_req = PCG_LOOP_AUTO;      // requested solve loop
  int az_req = PCG_AZ_AUTO;          // requested form of A z in the stencil sweep
  // multigrid preconditioner (row-tiled layout): levels 1..L-1 (level 0 is
  // the solver's own grid), the finest level's two iterates, and the number
  // of kernels one V-cycle launches
  int prec = PCG_PREC_LINE;
  int mg_nu = 1, mg_max_levels = 0;
  double mg_omega = 0.8;
  std::vector<pcg::MgLevel> mg;
  double *mg_x0 = nullptr, *mg_y0 = nullptr;
  int mg_grid_first = 1, mg_grid_smooth = 1;
  int mg_launches = 0;
  // host copies of the scalar coefficients, from which the coarse levels'
  // tables are built (a_h is averaged on the device)
  std::vector<double> dz_host;
  double a_h_host = 0.0, a_v_host = 0.0, mass_host = 0.0;
  int grid_ps = 0;                   // blocks of the persistent loop (0: not available)
  int cl_ctas = 0;                   // CTAs of the cluster loop (0: does not fit)
  unsigned int test_absent = 0;      // test hook: arrivals the persistent barriers miss
  size_t partials_cap = 0;           // doubles in `partials`
  // CUDA graphs of the row-tiled loop, one set without and one with timing
  // events ([timing]); each set has two instances, launched alternately so
  // that one can be read back (timing) while the other runs.  A set is
  // captured again when config_gen or the batch size changed since its last
  // capture, so switching timing on and off costs no capture once both exist.
  BatchGraph graphs[2][2];
  cudaStream_t cap_stream = nullptr;  // private stream for the captures
  unsigned long long config_gen = 1;  // bumped by every change a graph depends on
  unsigned long long graph_gen[2] = {0, 0};
  int graph_batch[2] = {0, 0};
  bool graphs_off = false;            // a capture failed: direct launches from then on
  int hist_cap = 0;
  DevState* state = nullptr;
  double *b_host_api = nullptr, *x_host_api = nullptr;  // device copies for pcg_solve_host
  // device address of the fixed scratch array of pcg_precond_dot_noalloc (not
  // an allocation of the context: the array lives in the library's module)
  double* noalloc_partials = nullptr;
  // the tensor-memory column solves (pcg_tmem.cu) can be launched; tmem_off:
  // switched off by the test hook pcg_test_tensor_memory
  bool tmem_ok = false, tmem_off = false;
  // second stream of pcg_update_solve_host: b and x0 go in while the set-up runs
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t copy_done = nullptr;
  // pcg_update_solve_host_async: x of consecutive calls alternates between two
  // device copies (x_host_api and x_async2); its copy-out runs on out_stream
  // and out_done[k] marks the end of the last one that read copy k
  double* x_async2 = nullptr;
  cudaStream_t out_stream = nullptr;
  cudaEvent_t out_done[2] = {nullptr, nullptr}, solved = nullptr;
  bool out_pending[2] = {false, false};
  const double* out_host[2] = {nullptr, nullptr};  // the host buffer each copy-out writes
  int out_slot = 0;
  // set by the host-buffer entry points right before their solve (and taken
  // back at its start): the initial guess is zero and its device copy was not
  // written, so the row-tiled start reads no x
  bool x0_zero = false;
  DevState* pinned = nullptr;                           // 3 host slots
  // flags the set-up kernels write straight into host memory (mapped, page-
  // locked): [0] the a_h field check, [1] the pivots of the Thomas factors.
  // A device-to-host copy would queue behind an asynchronous call's copy-out
  // of x on the same copy engine (1 GB, 5.6 ms); a kernel's store does not.
  int* hflags = nullptr;
  int* dflags = nullptr;  // the device's address of hflags
  // page-locked copy of the per-level table being uploaded, and the end of
  // that upload (the next update waits for it before it writes the copy)
  double* lev_pinned = nullptr;
  cudaEvent_t lev_done = nullptr;
  int grid_m = 1, grid_a = 1;
  long long last_launches = 0;
  // timing
  bool timing = false;
  std::vector<KernelEvent> events;  // recorded during the current solve
  std::vector<cudaEvent_t> event_pool;
  size_t pool_used = 0;
  double ms[PCG_K_COUNT] = {0};
  long long launches[PCG_K_COUNT] = {0};
  std::string err = "no error";
};

namespace {

int fail(pcg_ctx* ctx, int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (ctx)
    ctx->err = buf;
  else
    g_create_error = buf;
  return status;
}

int cuda_fail(pcg_ctx* ctx, cudaError_t e, const char* what) {
  // a failed runtime call also leaves its error as the thread's last error;
  // taken back here, so that the next launch check of this or another context
  // does not see it (a sticky error stays with the device whatever this does)
  (void)cudaGetLastError();
  const int st = (e == cudaErrorMemoryAllocation) ? PCG_ENOMEM : PCG_ECUDA;
  return fail(ctx, st, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (ok && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool finite_nonneg(double v) { return std::isfinite(v) && v >= 0.0; }

// PCG_EINVAL naming the first value of an a_h field that is not finite and
// >= 0, or PCG_OK.
int first_bad_field_value(pcg_ctx* ctx, const double* f, long long n) {
  for (long long i = 0; i < n; ++i)
    if (!finite_nonneg(f[i]))
      return fail(ctx, PCG_EINVAL, "a_h_field[%lld] must be finite and >= 0", i);
  return PCG_OK;
}

// field_on_device: the a_h field is checked by load_coeffs on the device
// (its staging copy) instead of here.
int validate_coeffs(pcg_ctx* ctx, int nx, int ny, int nz, const pcg_coeffs* c,
                    bool field_on_device = false) {
  if (!c) return fail(ctx, PCG_EINVAL, "coeffs is NULL");
  if (!finite_nonneg(c->a_v)) return fail(ctx, PCG_EINVAL, "a_v must be finite and >= 0");
  if (!(std::isfinite(c->mass) && c->mass > 0.0))
    return fail(ctx, PCG_EINVAL, "mass must be finite and > 0");
  if (!c->a_h_field && !finite_nonneg(c->a_h))
    return fail(ctx, PCG_EINVAL, "a_h must be finite and >= 0");
  if (c->a_h_field && !field_on_device) {
    const int st = first_bad_field_value(ctx, c->a_h_field, (long long)nx * ny);
    if (st) return st;
  }
  if (c->dz)
    for (int k = 0; k < nz; ++k)
      if (!(std::isfinite(c->dz[k]) && c->dz[k] > 0.0))
        return fail(ctx, PCG_EINVAL, "dz[%d] must be finite and > 0", k);
  return PCG_OK;
}

// Per-level tables (eq. (17): the vertical discretisation is the same in
// every column and only nz long).  For a constant a_h the Thomas factors are
// identical in every column and are computed here once.
//
// `area` is the horizontal cell area (1 on the solver's grid, 4^l on
// multigrid level l): the zero-order and vertical terms are integrated over
// it, the horizontal face weights keep their form.  Powers of two scale
// exactly, so a level's table is the area times the unit one, bit for bit.
int build_levels(pcg_ctx* ctx, int nz, const pcg_coeffs* c, bool varying,
                 std::vector<double>& lev, double area = 1.0) {
  using namespace pcg;
  lev.assign((size_t)kLevCount * nz, 0.0);
  std::vector<double> h(nz), tup(nz), tdn(nz);
  for (int k = 0; k < nz; ++k) h[k] = c->dz ? c->dz[k] : 1.0;
  for (int k = 0; k < nz; ++k)
    tup[k] = (k < nz - 1) ? c->a_v / (0.5 * (h[k] + h[k + 1])) * area : 0.0;
  for (int k = 0; k < nz; ++k) tdn[k] = (k > 0) ? tup[k - 1] : 0.0;
  double nphi_prev = 0.0;
  for (int k = 0; k < nz; ++k) {
    const double base = c->mass * h[k] * area + tup[k] + tdn[k];
    lev[LV_UP * nz + k] = -tup[k];
    lev[LV_DN * nz + k] = -tdn[k];
    lev[LV_H * nz + k] = h[k];
    lev[LV_TUP * nz + k] = tup[k];
    lev[LV_TDN * nz + k] = tdn[k];
    if (varying) {
      lev[LV_DIAG * nz + k] = base;
      lev[LV_HW * nz + k] = -h[k];
    } else {
      const double diag = base + h[k] * (4.0 * c->a_h);
      lev[LV_DIAG * nz + k] = diag;
      lev[LV_HW * nz + k] = -h[k] * c->a_h;
      const double D = diag - tdn[k] * nphi_prev;
      if (!(D > 0.0) || !std::isfinite(D))
        return fail(ctx, PCG_EBREAKDOWN, "Thomas pivot D_%d = %g is not positive", k, D);
      lev[LV_NPHI * nz + k] = tup[k] / D;
      lev[LV_INVD * nz + k] = 1.0 / D;
      nphi_prev = tup[k] / D;
    }
  }
  return PCG_OK;
}

template <typename T>
cudaError_t dalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
}

void mg_release(pcg_ctx* ctx);

void free_all(pcg_ctx* ctx) {
  double* bufs[] = {ctx->r,     ctx->z,     ctx->p,     ctx->q,        ctx->lev,
                    ctx->ah,    ctx->ah_stage, ctx->faceE, ctx->faceN, ctx->cdiag,  ctx->tnphi,
                    ctx->tinvd, ctx->partials, ctx->hist, ctx->b_host_api, ctx->x_host_api,
                    ctx->x_async2,
                    ctx->wscratch, ctx->u_t, ctx->cdiag_t, ctx->cwE_t, ctx->cwN_t,
                    ctx->nscratch,
                    ctx->op.sp_nphi, ctx->op.sp_invd, ctx->op.sp_ta, ctx->op.sp_tb,
                    ctx->op.sp_corners, ctx->op.sp_invdS, ctx->op.sp_nphiS};
  for (double* b : bufs)
    if (b) cudaFree(b);
  if (ctx->state) cudaFree(ctx->state);
  if (ctx->pinned) cudaFreeHost(ctx->pinned);
  if (ctx->hflags) cudaFreeHost(ctx->hflags);
  if (ctx->lev_pinned) cudaFreeHost(ctx->lev_pinned);
  if (ctx->lev_done) cudaEventDestroy(ctx->lev_done);
  ctx->lev_done = nullptr;
  for (cudaEvent_t e : ctx->event_pool) cudaEventDestroy(e);
  ctx->event_pool.clear();
  for (auto& set : ctx->graphs)
    for (BatchGraph& g : set) {
      if (g.exec) cudaGraphExecDestroy(g.exec);
      g.exec = nullptr;
      for (cudaEvent_t e : g.ev) cudaEventDestroy(e);
      g.ev.clear();
    }
  if (ctx->cap_stream) cudaStreamDestroy(ctx->cap_stream);
  ctx->cap_stream = nullptr;
  if (ctx->copy_done) cudaEventDestroy(ctx->copy_done);
  ctx->copy_done = nullptr;
  if (ctx->copy_stream) cudaStreamDestroy(ctx->copy_stream);
  ctx->copy_stream = nullptr;
  for (cudaEvent_t& ev : ctx->out_done) {
    if (ev) cudaEventDestroy(ev);
    ev = nullptr;
  }
  if (ctx->solved) cudaEventDestroy(ctx->solved);
  ctx->solved = nullptr;
  if (ctx->out_stream) cudaStreamDestroy(ctx->out_stream);
  ctx->out_stream = nullptr;
  mg_release(ctx);
}

// The set-up kernels' pivot flag (DevState::setup_error) on the host, after
// the stream's work so far: a kernel stores it into mapped host memory
// (hflags[1]), so the wait involves no copy engine (see pcg_ctx::hflags).
cudaError_t read_setup_error(pcg_ctx* ctx, int* bad) {
  volatile int* hf = ctx->hflags;
  hf[1] = 0;
  cudaError_t e = pcg::launch_flag_to_host(&ctx->state->setup_error, ctx->dflags + 1, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  *bad = hf[1];
  return e;
}

// Tables of the substructured column solve for the current coefficients.
// Synchronous.
int run_split_setup(pcg_ctx* ctx) {
  cudaError_t e = cudaMemsetAsync(&ctx->state->setup_error, 0, sizeof(int), ctx->stream);
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  if (ctx->timing) {
    cudaEventCreate(&t0);
    cudaEventCreate(&t1);
    if (t0) cudaEventRecord(t0, ctx->stream);
  }
  if (e == cudaSuccess) e = pcg::launch_split_setup(ctx->op, ctx->split_p, ctx->state, ctx->stream);
  if (t1) cudaEventRecord(t1, ctx->stream);
  int bad = 0;
  if (e == cudaSuccess) e = read_setup_error(ctx, &bad);
  if (t0 && t1) {
    float ms = 0.0f;
    if (e == cudaSuccess && cudaEventElapsedTime(&ms, t0, t1) == cudaSuccess) {
      ctx->ms[PCG_K_SETUP] += ms;
      ctx->launches[PCG_K_SETUP] += 2;
    }
  }
  if (t0) cudaEventDestroy(t0);
  if (t1) cudaEventDestroy(t1);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "substructuring set-up");
  if (bad) return fail(ctx, PCG_EBREAKDOWN, "a pivot of the substructured column solve is not positive");
  return PCG_OK;
}

// ------------------------------------------------ multigrid levels
//
// Level l+1 merges the 2x2 columns of level l (nx, ny even), keeps the nz
// layers, and is eqs. (5)-(8) on cells of horizontal area 4^(l+1) with a_h
// averaged over the merged columns.  Coarsening stops when nx or ny is odd,
// or at mg_max_levels levels (0: no cap).
int mg_count_levels(int nx, int ny, int max_levels) {
  int L = 1;
  while ((max_levels <= 0 || L < max_levels) && nx % 2 == 0 && ny % 2 == 0) {
    nx /= 2;
    ny /= 2;
    ++L;
  }
  return L;
}

void mg_release(pcg_ctx* ctx) {
  for (pcg::MgLevel& m : ctx->mg) {
    double* bufs[] = {m.lev,   m.ah,    m.faceE, m.faceN, m.cdiag, m.cdiag_t, m.cwE_t,
                      m.cwN_t, m.tnphi, m.tinvd, m.b,     m.x,     m.y};
    for (double* b : bufs)
      if (b) cudaFree(b);
  }
  ctx->mg.clear();
  if (ctx->mg_x0) cudaFree(ctx->mg_x0);
  if (ctx->mg_y0) cudaFree(ctx->mg_y0);
  ctx->mg_x0 = ctx->mg_y0 = nullptr;
}

// Allocate the coarse levels and the finest level's iterates.
int mg_allocate(pcg_ctx* ctx) {
  mg_release(ctx);
  const Op& f = ctx->op;
  const int L = mg_count_levels(f.nx, f.ny, ctx->mg_max_levels);
  if (L < 2)
    return fail(ctx, PCG_EINVAL, "multigrid needs a grid with even nx and ny (got %d x %d)", f.nx,
                f.ny);
  const bool fields = ctx->has_field_buffers;
  cudaError_t e = dalloc(&ctx->mg_x0, (size_t)f.ntiles * pcg::kTile * f.nz);
  if (e == cudaSuccess) e = dalloc(&ctx->mg_y0, (size_t)f.ntiles * pcg::kTile * f.nz);
  int nx = f.nx, ny = f.ny;
  ctx->mg.resize(L - 1);
  for (int l = 1; l < L && e == cudaSuccess; ++l) {
    nx /= 2;
    ny /= 2;
    pcg::MgLevel& m = ctx->mg[l - 1];
    Op& o = m.op;
    o = Op{};
    o.nx = nx;
    o.ny = ny;
    o.nz = f.nz;
    o.ncols = (long long)nx * ny;
    o.n = o.ncols * f.nz;
    o.ntiles = (o.ncols + pcg::kTile - 1) / pcg::kTile;
    const size_t npad = (size_t)o.ntiles * pcg::kTile * f.nz;
    e = dalloc(&m.lev, (size_t)pcg::kLevCount * f.nz);
    if (e == cudaSuccess) e = dalloc(&m.b, npad);
    if (e == cudaSuccess) e = dalloc(&m.x, npad);
    if (e == cudaSuccess) e = dalloc(&m.y, npad);
    if (e == cudaSuccess && fields) {
      e = dalloc(&m.ah, o.ncols);
      if (e == cudaSuccess) e = dalloc(&m.faceE, o.ncols);
      if (e == cudaSuccess) e = dalloc(&m.faceN, o.ncols);
      if (e == cudaSuccess) e = dalloc(&m.cdiag, o.n);
      if (e == cudaSuccess) e = dalloc(&m.cdiag_t, npad);
      if (e == cudaSuccess) e = dalloc(&m.cwE_t, npad);
      if (e == cudaSuccess) e = dalloc(&m.cwN_t, npad);
      if (e == cudaSuccess) e = dalloc(&m.tnphi, npad);
      if (e == cudaSuccess) e = dalloc(&m.tinvd, npad);
    }
    o.lev = m.lev;
    o.ah = m.ah;
    o.faceE = m.faceE;
    o.faceN = m.faceN;
    o.cdiag = m.cdiag;
    o.cdiag_t = m.cdiag_t;
    o.cwE_t = m.cwE_t;
    o.cwN_t = m.cwN_t;
    o.tnphi = m.tnphi;
    o.tinvd = m.tinvd;
  }
  if (e != cudaSuccess) {
    mg_release(ctx);
    return cuda_fail(ctx, e, "multigrid level allocation");
  }
  return PCG_OK;
}

// Coarse level tables for the current coefficients, and the grids of the
// Thomas sweeps on every level.  The per-level tables come from the host
// copies of the scalar coefficients; a_h is averaged level by level on the
// device.  Synchronous (one wait, for the pivot check).
int mg_setup(pcg_ctx* ctx) {
  const Op& f = ctx->op;
  const bool varying = f.varying != 0;
  pcg_coeffs c{};
  c.a_h = ctx->a_h_host;
  c.a_v = ctx->a_v_host;
  c.mass = ctx->mass_host;
  c.dz = ctx->dz_host.data();
  double area = 1.0;
  cudaError_t e = cudaMemsetAsync(&ctx->state->setup_error, 0, sizeof(int), ctx->stream);
  for (size_t l = 0; l < ctx->mg.size() && e == cudaSuccess; ++l) {
    pcg::MgLevel& m = ctx->mg[l];
    Op& o = m.op;
    const Op& fine = l ? ctx->mg[l - 1].op : f;
    area *= 4.0;
    o.varying = varying ? 1 : 0;
    std::vector<double> lev;
    int st = build_levels(ctx, f.nz, &c, varying, lev, area);
    if (st) return st;
    // (a pageable source: the call returns once the table is staged)
    e = cudaMemcpyAsync(m.lev, lev.data(), lev.size() * sizeof(double), cudaMemcpyHostToDevice,
                        ctx->stream);
    if (e == cudaSuccess && varying) {
      e = pcg::launch_mg_coarse_ah(fine, o, fine.ah, m.ah, ctx->num_sms, ctx->stream);
      if (e == cudaSuccess) e = pcg::launch_face_coeffs(o, m.faceE, m.faceN, ctx->stream);
      if (e == cudaSuccess)
        e = pcg::launch_column_setup(o, ctx->state, m.cdiag, m.cdiag_t, m.cwE_t, m.cwN_t,
                                     m.tnphi, m.tinvd, ctx->stream);
    }
    m.grid_first = pcg::grid_mg_first(o, ctx->num_sms);
    m.grid_smooth = pcg::grid_mg_smooth(o, ctx->num_sms);
  }
  ctx->mg_grid_first = pcg::grid_mg_first(f, ctx->num_sms);
  ctx->mg_grid_smooth = pcg::grid_mg_smooth(f, ctx->num_sms);
  int bad = 0;
  if (e == cudaSuccess) e = read_setup_error(ctx, &bad);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "multigrid level set-up");
  if (bad) return fail(ctx, PCG_EBREAKDOWN, "a Thomas pivot on a multigrid level is not positive");
  // reduction partials for the finest level's fused sweeps
  const size_t need = 2 * (size_t)std::max(ctx->mg_grid_first, ctx->mg_grid_smooth);
  if (need > ctx->partials_cap) {
    double* np = nullptr;
    e = dalloc(&np, need);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "reduction partials");
    cudaFree(ctx->partials);
    ctx->partials = np;
    ctx->partials_cap = need;
  }
  ctx->config_gen++;
  return PCG_OK;
}

// Enqueue one V-cycle, out = B b on the solver's grid (op0, row-tiled).
// fused: b is the solver's r, updated first (r <- r - alpha q), and the last
// smoothing step takes the scalar step of Algorithm 1.  *launches receives
// the number of kernels enqueued.
cudaError_t mg_enqueue(pcg_ctx* ctx, const Op& op0, double* b0, double* out, bool fused,
                       cudaStream_t s, int* launches) {
  const int L = (int)ctx->mg.size() + 1;
  const double w = ctx->mg_omega;
  const int nu = ctx->mg_nu;
  DevState* st = ctx->state;
  int cnt = 0;
  auto lvl_op = [&](int l) -> const Op& { return l ? ctx->mg[l - 1].op : op0; };
  auto lvl_b = [&](int l) { return l ? ctx->mg[l - 1].b : b0; };
  auto lvl_x = [&](int l) { return l ? ctx->mg[l - 1].x : ctx->mg_x0; };
  auto lvl_y = [&](int l) { return l ? ctx->mg[l - 1].y : ctx->mg_y0; };
  auto g_first = [&](int l) { return l ? ctx->mg[l - 1].grid_first : ctx->mg_grid_first; };
  auto g_smooth = [&](int l) { return l ? ctx->mg[l - 1].grid_smooth : ctx->mg_grid_smooth; };
  std::vector<double*> cur(L, nullptr);
  cudaError_t e = cudaSuccess;
  // down: smoothing from zero, then the restricted residual
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    const Op& o = lvl_op(l);
    double* c = lvl_x(l);
    double* other = lvl_y(l);
    e = pcg::launch_mg_first(o, st, lvl_b(l), ctx->q, c, w, fused && l == 0, ctx->partials,
                             ctx->hist, g_first(l), s);
    ++cnt;
    for (int i = 1; i < nu && e == cudaSuccess; ++i) {
      e = pcg::launch_mg_smooth(o, st, lvl_b(l), c, other, w, false, ctx->partials, ctx->hist,
                                g_smooth(l), ctx->num_sms, s);
      cnt += 2;
      std::swap(c, other);
    }
    cur[l] = c;
    if (l + 1 < L && e == cudaSuccess) {
      e = pcg::launch_mg_restrict(o, lvl_op(l + 1), st, lvl_b(l), c, nu == 1, w, lvl_b(l + 1),
                                  ctx->num_sms, s);
      ++cnt;
    }
  }
  // up: coarse-grid correction, then smoothing; the finest level's last step
  // writes `out`
  for (int l = L - 2; l >= 0 && e == cudaSuccess; --l) {
    const Op& o = lvl_op(l);
    double* c = cur[l];
    double* other = (c == lvl_x(l)) ? lvl_y(l) : lvl_x(l);
    e = pcg::launch_mg_prolong(o, lvl_op(l + 1), st, c, cur[l + 1], ctx->num_sms, s);
    ++cnt;
    for (int i = 0; i < nu && e == cudaSuccess; ++i) {
      const bool last = (i == nu - 1);
      double* dst = (l == 0 && last) ? out : other;
      e = pcg::launch_mg_smooth(o, st, lvl_b(l), c, dst, w, fused && l == 0 && last,
                                ctx->partials, ctx->hist, g_smooth(l), ctx->num_sms, s);
      cnt += 2;
      other = c;
      c = dst;
    }
    cur[l] = c;
  }
  if (launches) *launches = cnt;
  return e;
}

// Upload coefficients and (for a field) rebuild the per-column and per-cell
// tables on the device.  With a field the call waits twice: for the field's
// check before anything changes, and for the set-up kernels' pivot check;
// with a constant a_h it only queues the level table.  `meanwhile`, when
// given, is called once the set-up work is enqueued and before the host
// waits for it: work it enqueues on another stream runs alongside the set-up.
int load_coeffs(pcg_ctx* ctx, const pcg_coeffs* c, bool varying,
                const std::function<cudaError_t()>& meanwhile = {}) {
  if (varying) {
    // The field goes to a staging copy and is checked there, on the device
    // (on the host the 8 MB of a 1024 x 1024 field took 0.42 ms of every
    // update, with the GPU idle); only a field that passes replaces the
    // context's, so a rejected one leaves the context as it was.
    const size_t bytes = ctx->op.ncols * sizeof(double);
    volatile int* hf = ctx->hflags;
    hf[0] = 0;
    cudaError_t e = cudaMemcpyAsync(ctx->ah_stage, c->a_h_field, bytes, cudaMemcpyHostToDevice,
                                    ctx->stream);
    if (e == cudaSuccess)
      e = pcg::launch_check_field(ctx->ah_stage, ctx->op.ncols, ctx->dflags, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "upload of a_h_field");
    if (hf[0]) {
      const int st = first_bad_field_value(ctx, c->a_h_field, ctx->op.ncols);
      return st ? st : fail(ctx, PCG_EINVAL, "a_h_field changed while it was read");
    }
    std::swap(ctx->ah, ctx->ah_stage);
    ctx->op.ah = ctx->ah;
  }
  ctx->config_gen++;  // the sweeps' template choice follows op.varying
  std::vector<double> lev;
  int st = build_levels(ctx, ctx->op.nz, c, varying, lev);
  if (st) return st;
  // host copies for the multigrid levels
  ctx->a_h_host = c->a_h;
  ctx->a_v_host = c->a_v;
  ctx->mass_host = c->mass;
  ctx->dz_host.assign((size_t)ctx->op.nz, 1.0);
  if (c->dz) ctx->dz_host.assign(c->dz, c->dz + ctx->op.nz);
  // the table goes up from a page-locked copy, so the upload is queued on the
  // stream without a wait for the host (a pageable source would make the copy
  // wait for the stream's earlier work first)
  cudaError_t e = cudaEventSynchronize(ctx->lev_done);  // the previous upload has read the copy
  if (e == cudaSuccess) {
    std::memcpy(ctx->lev_pinned, lev.data(), lev.size() * sizeof(double));
    e = cudaMemcpyAsync(ctx->lev, ctx->lev_pinned, lev.size() * sizeof(double),
                        cudaMemcpyHostToDevice, ctx->stream);
  }
  if (e == cudaSuccess) e = cudaEventRecord(ctx->lev_done, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "upload of the level table");
  if (ctx->op.varying != (varying ? 1 : 0)) {
    ctx->op.varying = varying ? 1 : 0;
    if (ctx->num_sms > 0) ctx->cl_ctas = pcg::cluster_ctas(ctx->op);  // the tables it holds
  }
  if (varying) {
    e = cudaMemsetAsync(&ctx->state->setup_error, 0, sizeof(int), ctx->stream);
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    if (ctx->timing) {
      cudaEventCreate(&t0);
      cudaEventCreate(&t1);
      if (t0) cudaEventRecord(t0, ctx->stream);
    }
    if (e == cudaSuccess) e = pcg::launch_face_coeffs(ctx->op, ctx->faceE, ctx->faceN, ctx->stream);
    if (e == cudaSuccess)
      e = pcg::launch_column_setup(ctx->op, ctx->state, ctx->cdiag, ctx->cdiag_t, ctx->cwE_t,
                                   ctx->cwN_t, ctx->tnphi, ctx->tinvd, ctx->stream);
    if (t1) cudaEventRecord(t1, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "coefficient set-up kernels");
    if (meanwhile) {
      e = meanwhile();
      if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
    }
    int bad = 0;
    if (e == cudaSuccess) e = read_setup_error(ctx, &bad);
    if (t0 && t1) {
      float ms = 0.0f;
      if (e == cudaSuccess && cudaEventElapsedTime(&ms, t0, t1) == cudaSuccess) {
        ctx->ms[PCG_K_SETUP] += ms;
        ctx->launches[PCG_K_SETUP] += 2;
      }
    }
    if (t0) cudaEventDestroy(t0);
    if (t1) cudaEventDestroy(t1);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "coefficient set-up");
    if (bad) return fail(ctx, PCG_EBREAKDOWN, "a Thomas pivot of some column is not positive");
  } else if (meanwhile) {
    // a constant a_h: the level table is all there is, queued on the stream
    e = meanwhile();
    if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
  }
  if (ctx->split_p > 1) {
    st = run_split_setup(ctx);
    if (st) return st;
  }
  if (ctx->prec == PCG_PREC_MULTIGRID) return mg_setup(ctx);
  return PCG_OK;
}

cudaEvent_t pool_event(pcg_ctx* ctx) {
  if (ctx->pool_used == ctx->event_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    ctx->event_pool.push_back(e);
  }
  return ctx->event_pool[ctx->pool_used++];
}

// Launch helper: records start/stop events when timing is on.
template <typename F>
cudaError_t timed(pcg_ctx* ctx, int kind, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (ctx->timing) {
    a = pool_event(ctx);
    b = pool_event(ctx);
    if (a && b) cudaEventRecord(a, ctx->stream);
  }
  cudaError_t e = launch();
  ctx->last_launches++;
  if (ctx->timing && a && b) {
    cudaEventRecord(b, ctx->stream);
    ctx->events.push_back({kind, a, b});
  }
  return e;
}

// After the stream has been synchronised: fold the recorded events into the
// per-kernel totals.  Sweeps enqueued after the device set its completion
// flag return at once; only the first `work_m` preconditioner sweeps and
// `work_a` SpMV sweeps did work, and only those are counted.
void collect_events(pcg_ctx* ctx, long long work_m, long long work_a) {
  long long seen_m = 0, seen_a = 0;
  for (const KernelEvent& ke : ctx->events) {
    // the first-iteration sweeps come first in launch order, counted with
    // the rest of their kind's work
    const bool sweep_m = ke.kind == PCG_K_PRECOND_FUSED || ke.kind == PCG_K_PRECOND_FIRST;
    const bool sweep_a = ke.kind == PCG_K_SPMV_FUSED || ke.kind == PCG_K_SPMV_FIRST;
    if (sweep_m && seen_m++ >= work_m) continue;
    if (sweep_a && seen_a++ >= work_a) continue;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, ke.start, ke.stop) == cudaSuccess) {
      ctx->ms[ke.kind] += ms;
      ctx->launches[ke.kind]++;
    }
  }
  ctx->events.clear();
  ctx->pool_used = 0;
}

bool overlap(const double* a, const double* b, long long n) {
  return (a < b + n) && (b < a + n);
}
// [a, a+na) and [b, b+nb) share an element
bool overlap(const double* a, long long na, const double* b, long long nb) {
  return (a < b + nb) && (b < a + na);
}

// Grids that the automatic loop choice runs persistent (and the layout the
// automatic choices assume: row-tiled): fewer than 4 tiles of 32 columns per
// SM, where the batched sweeps are launch-bound, and up to 16 per SM while the
// grid has at most 6 M cells, where the persistent loop's 16 warps per SM
// still beat the batched sweeps (256x256x64: 137 against 146 us per
// iteration; at 384x384x64 the two are level).
bool persistent_grid(const pcg_ctx* ctx) {
  const long long nt = ctx->op.ntiles, sms = ctx->num_sms;
  return ctx->grid_ps > 0 && (nt < 4 * sms || (nt < 16 * sms && ctx->op.n <= (6LL << 20)));
}

// The loop the next solve runs (PCG_LOOP_BATCHED, PCG_LOOP_PERSISTENT or
// PCG_LOOP_CLUSTER).
int resolved_az(const pcg_ctx* ctx);
int resolved_loop(const pcg_ctx* ctx) {
  const bool eligible = ctx->layout == PCG_LAYOUT_TILED && ctx->split_p == 1 &&
                        ctx->prec == PCG_PREC_LINE &&
                        !(ctx->op.varying && ctx->factors == PCG_FACTORS_RECOMPUTE);
  if (!eligible || ctx->loop_req == PCG_LOOP_BATCHED) return PCG_LOOP_BATCHED;
  const bool cluster = ctx->cl_ctas > 0 && resolved_az(ctx) == PCG_AZ_RESIDUAL;
  if ((ctx->loop_req == PCG_LOOP_CLUSTER || ctx->loop_req == PCG_LOOP_AUTO) && cluster)
    return PCG_LOOP_CLUSTER;
  if (ctx->grid_ps > 0 && (ctx->loop_req == PCG_LOOP_PERSISTENT || persistent_grid(ctx) ||
                           ctx->loop_req == PCG_LOOP_CLUSTER))
    return PCG_LOOP_PERSISTENT;
  return PCG_LOOP_BATCHED;
}

// The form of A z that the next solve's stencil sweeps use (PCG_AZ_STENCIL
// or PCG_AZ_RESIDUAL): the residual form needs the Thomas column solve, whose
// z the sweep pairs with r (no substructuring, no multigrid).
int resolved_az(const pcg_ctx* ctx) {
  const bool split = ctx->layout == PCG_LAYOUT_TILED && ctx->split_p > 1;
  const bool eligible = !split && ctx->prec == PCG_PREC_LINE;
  return (eligible && ctx->az_req != PCG_AZ_STENCIL) ? PCG_AZ_RESIDUAL : PCG_AZ_STENCIL;
}

// The two sweeps of one iteration of the row-tiled loop, enqueued on `s`;
// with `ev`, boundary events before the first and between the two.
cudaError_t launch_tiled_iteration(pcg_ctx* ctx, const Op& op, bool split, int grid_pm,
                                   cudaStream_t s, cudaEvent_t* ev) {
  cudaError_t e = cudaSuccess;
  if (ev) e = cudaEventRecordWithFlags(ev[0], s, cudaEventRecordExternal);
  if (e == cudaSuccess) {
    if (ctx->prec == PCG_PREC_MULTIGRID)
      e = mg_enqueue(ctx, op, ctx->r, ctx->z, true, s, &ctx->mg_launches);
    else if (split)
      e = pcg::launch_precond_split(op, ctx->split_p, ctx->state, ctx->r, ctx->q, ctx->z,
                                    ctx->partials, ctx->hist, grid_pm, s);
    else
      e = pcg::launch_precond_tiled(op, ctx->state, ctx->r, ctx->q, ctx->z, ctx->partials,
                                    ctx->hist, grid_pm, s);
  }
  if (e == cudaSuccess && ev) e = cudaEventRecordWithFlags(ev[1], s, cudaEventRecordExternal);
  if (e == cudaSuccess)
    e = pcg::launch_spmv_tiled(op, ctx->state, ctx->z, ctx->r, ctx->u_t, ctx->p, ctx->q,
                               ctx->partials + 2 * grid_pm, ctx->grid_ta, s);
  return e;
}

// Capture `iters` iterations of the row-tiled loop into g (on the private
// capture stream; the graph is later launched on the context's stream).
cudaError_t capture_batch(pcg_ctx* ctx, const Op& op, bool split, int grid_pm, int iters,
                          bool timing, BatchGraph& g) {
  cudaError_t e = cudaSuccess;
  if (!ctx->cap_stream) e = cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  if (g.exec) cudaGraphExecDestroy(g.exec);
  g.exec = nullptr;
  if (timing) {
    while (e == cudaSuccess && g.ev.size() < 2 * (size_t)iters + 1) {
      cudaEvent_t ev = nullptr;
      e = cudaEventCreate(&ev);
      if (e == cudaSuccess) g.ev.push_back(ev);
    }
    if (e != cudaSuccess) return e;
  }
  e = cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < iters && e == cudaSuccess; ++i)
    e = launch_tiled_iteration(ctx, op, split, grid_pm, ctx->cap_stream,
                               timing ? &g.ev[2 * (size_t)i] : nullptr);
  if (e == cudaSuccess && timing)
    e = cudaEventRecordWithFlags(g.ev[2 * (size_t)iters], ctx->cap_stream,
                                 cudaEventRecordExternal);
  cudaGraph_t graph = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(ctx->cap_stream, &graph);
  if (e == cudaSuccess) e = ee;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&g.exec, graph, 0);
  if (graph) cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    g.exec = nullptr;
    (void)cudaGetLastError();
  }
  return e;
}

// Elapsed times of the sweeps of one finished batch graph, in launch order.
void read_batch_times(const BatchGraph& g, int iters, std::vector<float>& tm_m,
                      std::vector<float>& tm_a) {
  for (int i = 0; i < iters; ++i) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, g.ev[2 * i], g.ev[2 * i + 1]) == cudaSuccess) tm_m.push_back(ms);
    if (cudaEventElapsedTime(&ms, g.ev[2 * i + 1], g.ev[2 * i + 2]) == cudaSuccess) tm_a.push_back(ms);
  }
}

int solve_device(pcg_ctx* ctx, const double* b, double* x, double rtol, int maxit,
                 int* iters_out, double* res_hist) {
  const bool x0_zero_given = ctx->x0_zero;
  ctx->x0_zero = false;
  cudaError_t e;
  if (maxit + 1 > ctx->hist_cap) {
    double* nh = nullptr;
    e = dalloc(&nh, (size_t)maxit + 1);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "allocation of the residual history");
    if (ctx->hist) cudaFree(ctx->hist);
    ctx->hist = nh;
    ctx->hist_cap = maxit + 1;
    ctx->config_gen++;
  }
  Op op = ctx->op;
  cudaStream_t s = ctx->stream;
  ctx->last_launches = 0;
  ctx->events.clear();
  ctx->pool_used = 0;
  const bool tiled = ctx->layout == PCG_LAYOUT_TILED;
  op.recompute = (tiled && op.varying && ctx->factors == PCG_FACTORS_RECOMPUTE) ? 1 : 0;
  op.az_resid = resolved_az(ctx) == PCG_AZ_RESIDUAL ? 1 : 0;
  const bool mgrid = tiled && ctx->prec == PCG_PREC_MULTIGRID;
  const bool split = tiled && ctx->split_p > 1 && !mgrid;
  const int grid_pm = split ? ctx->grid_sp : ctx->grid_tm;  // preconditioner sweep blocks
  op.nscratch = ctx->nscratch;
  // r = b - A x0, the solver's start; the row-tiled layout writes r, u = x0
  // and p = q = 0 at its own positions in the same launch.  On large grids a
  // pass over x0 first finds out whether it is all +0.0, so that the start
  // reads neither x0 nor its neighbours then (small grids: one launch less).
  // A zero initial guess that a host-buffer entry point did not copy in needs
  // no pass at all: the flag is cleared and x is never read.
  const bool x0_zero = x0_zero_given && tiled;
  const bool x0_check = tiled && (x0_zero || op.n >= (1LL << 22));
  if (x0_zero) {
    e = cudaMemsetAsync(&ctx->state->x0_nonzero, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "initial guess flag");
  } else if (x0_check) {
    e = timed(ctx, PCG_K_RESIDUAL,
              [&] { return pcg::launch_x0_nonzero(x, op.n, ctx->state, ctx->num_sms, s); });
    if (e != cudaSuccess) return cuda_fail(ctx, e, "initial guess check launch");
  }
  // Persistent loop: every iteration in one cooperative kernel; cluster loop:
  // every iteration in one cluster, the vectors in its shared memory.
  const int loop = resolved_loop(ctx);
  const bool persistent = loop == PCG_LOOP_PERSISTENT || loop == PCG_LOOP_CLUSTER;
  // The batched row-tiled loop with stored factors and Thomas column solves
  // runs its first iteration with the first-iteration sweeps (alpha = beta =
  // 0, p = q = 0 never read), so the start writes neither p nor q.
  const bool first_direct = tiled && !persistent && !mgrid && !split && !op.recompute;
  e = timed(ctx, PCG_K_RESIDUAL, [&] {
    return tiled ? pcg::launch_residual_tiled(op, ctx->state, b, x, ctx->r, ctx->u_t, ctx->p,
                                              ctx->q, rtol, maxit, x0_check, s, !first_direct)
                 : pcg::launch_residual(op, ctx->state, b, x, ctx->r, ctx->p, ctx->q, rtol,
                                        maxit, ctx->grid_a, s);
  });
  if (e != cudaSuccess) return cuda_fail(ctx, e, "residual kernel launch");

  if (loop == PCG_LOOP_CLUSTER) {
    e = timed(ctx, PCG_K_LOOP, [&] {
      return pcg::launch_cluster_loop(op, ctx->state, ctx->r, ctx->u_t, ctx->p, ctx->hist,
                                      ctx->cl_ctas, s);
    });
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cluster solve loop launch");
  } else if (persistent) {
    e = timed(ctx, PCG_K_LOOP, [&] {
      return pcg::launch_persistent(op, ctx->state, ctx->r, ctx->q, ctx->z, ctx->u_t, ctx->p,
                                    ctx->partials, ctx->hist, ctx->grid_ps, ctx->test_absent,
                                    s);
    });
    if (e != cudaSuccess) return cuda_fail(ctx, e, "persistent solve loop launch");
  }

  // Enqueue the loop in batches; poll the device's `done` flag one batch
  // behind, so the GPU always has queued work and never waits for the host.
  const int batch = (op.n >= (1LL << 24)) ? 4 : 16;
  int enq = 0, slot = 0, pending = -1;
  cudaEvent_t ev[2] = {pool_event(ctx), pool_event(ctx)};
  if (!ev[0] || !ev[1]) return fail(ctx, PCG_ECUDA, "event creation failed");
  if (first_direct) {  // iteration 0, outside the graphs
    e = timed(ctx, PCG_K_PRECOND_FIRST, [&] {
      return pcg::launch_precond_tiled(op, ctx->state, ctx->r, ctx->q, ctx->z, ctx->partials,
                                       ctx->hist, grid_pm, s, true);
    });
    if (e == cudaSuccess && maxit > 0)
      e = timed(ctx, PCG_K_SPMV_FIRST, [&] {
        return pcg::launch_spmv_tiled(op, ctx->state, ctx->z, ctx->r, ctx->u_t, ctx->p, ctx->q,
                                      ctx->partials + 2 * grid_pm, ctx->grid_ta, s, true);
      });
    if (e != cudaSuccess) return cuda_fail(ctx, e, "first iteration launch");
    enq = 1;
  }
  bool stop = false;
  // Row-tiled layout: every batch is one launch of a CUDA graph (all its
  // operands are the context's own buffers).  Sweeps past the last
  // iteration see `done` and return at once, so every batch is a full one.
  bool use_graphs = tiled && !ctx->graphs_off && !persistent;
  const int tv = ctx->timing ? 1 : 0;
  BatchGraph* graphs = ctx->graphs[tv];
  if (use_graphs && (ctx->graph_gen[tv] != ctx->config_gen || ctx->graph_batch[tv] != batch)) {
    for (BatchGraph* g = graphs; g != graphs + 2; ++g) {
      if (capture_batch(ctx, op, split, grid_pm, batch, ctx->timing, *g) != cudaSuccess) {
        use_graphs = false;
        ctx->graphs_off = true;  // this driver or device refuses: launch directly from now on
        break;
      }
    }
    ctx->graph_gen[tv] = ctx->config_gen;
    ctx->graph_batch[tv] = batch;
  }
  std::vector<float> tm_m, tm_a;  // graph sweep times in launch order (timing)
  while (use_graphs && enq <= maxit && !stop) {
    e = cudaGraphLaunch(graphs[slot].exec, s);
    ctx->last_launches += (long long)(mgrid ? ctx->mg_launches + 1 : 2) * batch;
    enq += batch;
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(&ctx->pinned[slot], ctx->state, sizeof(DevState),
                          cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[slot], s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "solve batch launch");
    if (pending >= 0) {
      e = cudaEventSynchronize(ev[pending]);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "solve loop");
      if (ctx->timing) read_batch_times(graphs[pending], batch, tm_m, tm_a);
      if (ctx->pinned[pending].done) stop = true;
    }
    pending = slot;
    slot ^= 1;
  }
  const int last_graph = (use_graphs && pending >= 0) ? pending : -1;  // read after the final sync
  if (use_graphs || persistent) stop = true;
  while (enq <= maxit && !stop) {
    const int nb = std::min(batch, maxit + 1 - enq);
    for (int i = 0; i < nb; ++i) {
      e = timed(ctx, PCG_K_PRECOND_FUSED, [&] {
        if (mgrid) {
          cudaError_t ee = mg_enqueue(ctx, op, ctx->r, ctx->z, true, s, &ctx->mg_launches);
          ctx->last_launches += ctx->mg_launches - 1;  // timed() counts one
          return ee;
        }
        if (split)
          return pcg::launch_precond_split(op, ctx->split_p, ctx->state, ctx->r, ctx->q, ctx->z,
                                           ctx->partials, ctx->hist, ctx->grid_sp, s);
        if (tiled)
          return pcg::launch_precond_tiled(op, ctx->state, ctx->r, ctx->q, ctx->z,
                                           ctx->partials, ctx->hist, grid_pm, s);
        // column layout: the tensor-memory sweep where it applies (nz = 32, 64,
        // 128); its grid is smaller than grid_m, so the stencil sweep's
        // partials after 2*grid_m stay clear of its own
        if (ctx->tmem_ok && !ctx->tmem_off && pcg::precond_tmem_supported(op, ctx->r, ctx->q, ctx->z))
          return pcg::launch_precond_tmem(op, ctx->state, ctx->r, ctx->q, ctx->z, ctx->partials,
                                          ctx->hist, true,
                                          pcg::grid_precond_tmem(ctx->op, ctx->num_sms), s);
        return pcg::launch_precond_fused(op, ctx->state, ctx->r, ctx->q, ctx->z, ctx->partials,
                                         ctx->hist, ctx->grid_m, s);
      });
      if (e != cudaSuccess) return cuda_fail(ctx, e, "preconditioner sweep launch");
      if (enq + i < maxit) {
        e = timed(ctx, PCG_K_SPMV_FUSED, [&] {
          return tiled ? pcg::launch_spmv_tiled(op, ctx->state, ctx->z, ctx->r, ctx->u_t, ctx->p,
                                                ctx->q,
                                                ctx->partials + 2 * grid_pm, ctx->grid_ta, s)
                       : pcg::launch_spmv_fused(op, ctx->state, ctx->z, ctx->r, x, ctx->p,
                                                ctx->q, ctx->partials + 2 * ctx->grid_m,
                                                ctx->grid_a, s);
        });
        if (e != cudaSuccess) return cuda_fail(ctx, e, "SpMV sweep launch");
      }
    }
    enq += nb;
    e = cudaMemcpyAsync(&ctx->pinned[slot], ctx->state, sizeof(DevState),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[slot], s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "state poll");
    if (pending >= 0) {
      e = cudaEventSynchronize(ev[pending]);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "solve loop");
      if (ctx->pinned[pending].done) stop = true;
    }
    pending = slot;
    slot ^= 1;
  }
  e = timed(ctx, PCG_K_FINALIZE, [&] {
    return tiled ? pcg::launch_from_tiled(op, ctx->state, ctx->u_t, ctx->p, x, s)
                 : pcg::launch_finalize(op, ctx->state, x, ctx->p, ctx->grid_a, s);
  });
  if (e != cudaSuccess) return cuda_fail(ctx, e, "finalize launch");
  e = cudaMemcpyAsync(&ctx->pinned[2], ctx->state, sizeof(DevState), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "solve");
  const DevState fin = ctx->pinned[2];
  if (!fin.done) return fail(ctx, PCG_ECUDA, "solve ended without the device completion flag");
  if (res_hist && fin.iters >= 0) {
    e = cudaMemcpyAsync(res_hist, ctx->hist, sizeof(double) * ((size_t)fin.iters + 1),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "residual history copy");
  }
  if (ctx->timing) {
    collect_events(ctx, fin.it, fin.it > 0 ? fin.it - 1 : 0);
    if (last_graph >= 0) read_batch_times(graphs[last_graph], batch, tm_m, tm_a);
    // only the sweeps that did work: the first `it` preconditioner and
    // `it - 1` stencil sweeps in launch order (the graphs' after the directly
    // launched first iteration, which collect_events counted)
    const long long f = (first_direct && last_graph >= 0) ? 1 : 0;
    const size_t wm = std::min<size_t>(tm_m.size(), fin.it > f ? (size_t)(fin.it - f) : 0);
    const size_t wa =
        std::min<size_t>(tm_a.size(), fin.it > 1 + f ? (size_t)(fin.it - 1 - f) : 0);
    for (size_t i = 0; i < wm; ++i) ctx->ms[PCG_K_PRECOND_FUSED] += tm_m[i];
    for (size_t i = 0; i < wa; ++i) ctx->ms[PCG_K_SPMV_FUSED] += tm_a[i];
    ctx->launches[PCG_K_PRECOND_FUSED] += (long long)wm;
    ctx->launches[PCG_K_SPMV_FUSED] += (long long)wa;
  }
  if (iters_out) *iters_out = fin.iters;
  if (fin.status == PCG_ENOTCONV)
    return fail(ctx, PCG_ENOTCONV, "no convergence to rtol=%g in %d iterations (last ratio %g)",
                rtol, maxit, fin.R0 > 0 ? std::sqrt(fin.last_R / fin.R0) : 0.0);
  if (fin.status == PCG_ETIMEOUT || fin.dev_error)
    return fail(ctx, PCG_ETIMEOUT, "a bounded device wait ran out after %d iterations",
                fin.iters);
  if (fin.status == PCG_EBREAKDOWN)
    return fail(ctx, PCG_EBREAKDOWN,
                "breakdown after %d iterations: ||r||^2=%g <r,z>=%g <p,Ap>=%g", fin.iters,
                fin.last_R, fin.last_kappa, fin.last_sigma);
  return fin.status;
}

}  // namespace

extern "C" {

int pcg_create(int nx, int ny, int nz, const pcg_coeffs* coeffs, pcg_ctx** out) {
  if (!out) return fail(nullptr, PCG_EINVAL, "out is NULL");
  *out = nullptr;
  if (nx < 1 || ny < 1 || nz < 1)
    return fail(nullptr, PCG_EINVAL, "grid %d x %d x %d: every size must be >= 1", nx, ny, nz);
  const long long ncols = (long long)nx * ny;
  const long long n = ncols * nz;
  if (n >= (1LL << 40)) return fail(nullptr, PCG_EINVAL, "grid too large (%lld cells)", n);
  int st = validate_coeffs(nullptr, nx, ny, nz, coeffs);
  if (st) return st;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) {
    int count = 0;
    e = cudaGetDeviceCount(&count);
    if (e == cudaSuccess && count < 1) e = cudaErrorNoDevice;
  }
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "no usable CUDA device");

  pcg_ctx* ctx = new (std::nothrow) pcg_ctx();
  if (!ctx) return fail(nullptr, PCG_ENOMEM, "host allocation failed");
  ctx->device = dev;
  cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev);
  Op& op = ctx->op;
  op.nx = nx;
  op.ny = ny;
  op.nz = nz;
  op.pz = (nz + 15) / 16 * 16;
  op.pt = (nz % 4 == 0) ? nz + 2 : (nz % 2 == 0 ? nz : nz + 1);
  op.fixed = (nz == 32 || nz == 64 || nz == 128) ? 1 : 0;
  op.ncols = ncols;
  op.n = n;
  op.ntiles = (ncols + pcg::kTile - 1) / pcg::kTile;
  const bool varying = coeffs->a_h_field != nullptr;
  ctx->has_field_buffers = varying;

  auto bail = [&](int status) {
    std::string msg = ctx->err;
    free_all(ctx);
    delete ctx;
    g_create_error = msg;
    return status;
  };
  // internal vectors are sized for the row-tiled layout too (last tile padded)
  const long long npad = op.ntiles * pcg::kTile * nz;
  e = dalloc(&ctx->r, npad);
  if (e == cudaSuccess) e = dalloc(&ctx->z, npad);
  if (e == cudaSuccess) e = dalloc(&ctx->p, npad);
  if (e == cudaSuccess) e = dalloc(&ctx->q, npad);
  if (e == cudaSuccess) e = dalloc(&ctx->lev, (size_t)pcg::kLevCount * nz);
  if (e == cudaSuccess) e = dalloc(&ctx->state, 1);
  if (e == cudaSuccess) e = cudaMemset(ctx->state, 0, sizeof(DevState));
  if (e == cudaSuccess && varying) {
    const size_t tiled = (size_t)op.ntiles * pcg::kTile * nz;
    e = dalloc(&ctx->ah, ncols);
    if (e == cudaSuccess) e = dalloc(&ctx->ah_stage, ncols);
    if (e == cudaSuccess) e = dalloc(&ctx->faceE, ncols);
    if (e == cudaSuccess) e = dalloc(&ctx->faceN, ncols);
    if (e == cudaSuccess) e = dalloc(&ctx->cdiag, n);
    if (e == cudaSuccess) e = dalloc(&ctx->tnphi, tiled);
    if (e == cudaSuccess) e = dalloc(&ctx->tinvd, tiled);
  }
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&ctx->pinned), 3 * sizeof(DevState),
                      cudaHostAllocDefault);
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&ctx->hflags), 4 * sizeof(int), cudaHostAllocMapped);
  if (e == cudaSuccess)
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&ctx->dflags), ctx->hflags, 0);
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&ctx->lev_pinned),
                      (size_t)pcg::kLevCount * nz * sizeof(double), cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->lev_done, cudaEventDisableTiming);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "workspace allocation"));
  memset(ctx->pinned, 0, 3 * sizeof(DevState));
  op.lev = ctx->lev;
  op.ah = ctx->ah;
  op.faceE = ctx->faceE;
  op.faceN = ctx->faceN;
  op.cdiag = ctx->cdiag;
  op.tnphi = ctx->tnphi;
  op.tinvd = ctx->tinvd;
  op.varying = varying ? 1 : 0;

  e = pcg::prepare_kernels(op);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "kernel attribute set-up"));
  // the tensor-memory column solves need their shared-memory attribute; where
  // it cannot be set the other column-solve kernels run instead
  ctx->tmem_ok = pcg::prepare_precond_tmem() == cudaSuccess;
  (void)cudaGetLastError();
  op.tmem = ctx->tmem_ok ? 1 : 0;
  ctx->grid_m = pcg::grid_precond(op, ctx->num_sms);  // also sets op.stream_smem
  ctx->grid_a = pcg::grid_spmv(op, ctx->num_sms);
  ctx->grid_tm = pcg::grid_tiled_precond(op, ctx->num_sms);
  ctx->grid_ta = pcg::grid_tiled_spmv(op, ctx->num_sms);
  ctx->grid_ps = pcg::grid_persistent(op, ctx->num_sms);
  ctx->cl_ctas = pcg::cluster_ctas(op);
  ctx->partials_cap = 2 * (size_t)std::max(std::max(ctx->grid_m + ctx->grid_a,
                                                     ctx->grid_tm + ctx->grid_ta),
                                            2 * ctx->grid_ps);
  e = dalloc(&ctx->partials, ctx->partials_cap);
  if (e == cudaSuccess && op.fixed)
    e = dalloc(&ctx->wscratch, (size_t)ctx->grid_m * pcg::kTile * nz);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "workspace allocation"));
  op.wscratch = ctx->wscratch;
  // device address of the allocation-free entry point's fixed scratch array
  e = pcg::noalloc_scratch_address(&ctx->noalloc_partials);
  if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "scratch address lookup"));
  st = load_coeffs(ctx, coeffs, varying);
  if (st) return bail(st);
  st = pcg_set_layout(ctx, PCG_LAYOUT_TILED);  // the default solver layout
  if (st) return bail(st);
  st = pcg_set_substructuring(ctx, 0);  // automatic: only grids with few tiles
  if (st) return bail(st);
  *out = ctx;
  return PCG_OK;
}

void pcg_destroy(pcg_ctx* ctx) {
  if (!ctx) return;
  DeviceGuard g(ctx->device);
  cudaStreamSynchronize(ctx->stream);
  if (ctx->copy_stream) cudaStreamSynchronize(ctx->copy_stream);
  if (ctx->out_stream) cudaStreamSynchronize(ctx->out_stream);
  free_all(ctx);
  delete ctx;
}

int pcg_update_coeffs(pcg_ctx* ctx, const pcg_coeffs* coeffs) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  int st = validate_coeffs(ctx, ctx->op.nx, ctx->op.ny, ctx->op.nz, coeffs, true);
  if (st) return st;
  const bool varying = coeffs->a_h_field != nullptr;
  if (varying && !ctx->has_field_buffers)
    return fail(ctx, PCG_EINVAL,
                "context was created with a constant a_h; it cannot take an a_h field");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  return load_coeffs(ctx, coeffs, varying);
}

int pcg_set_layout(pcg_ctx* ctx, int layout) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (layout != PCG_LAYOUT_COLUMN && layout != PCG_LAYOUT_TILED)
    return fail(ctx, PCG_EINVAL, "unknown layout %d", layout);
  if (layout == ctx->layout) return PCG_OK;
  if (ctx->prec == PCG_PREC_MULTIGRID)
    return fail(ctx, PCG_EINVAL, "the multigrid preconditioner needs the row-tiled layout");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  const long long npad = ctx->op.ntiles * pcg::kTile * ctx->op.nz;
  if (e == cudaSuccess && layout == PCG_LAYOUT_TILED && !ctx->u_t) e = dalloc(&ctx->u_t, npad);
  if (e == cudaSuccess && layout == PCG_LAYOUT_TILED && ctx->has_field_buffers &&
      !(ctx->cdiag_t && ctx->cwE_t && ctx->cwN_t)) {
    // each table where it is missing: an earlier attempt that ran out of
    // memory may have made some of them
    for (double** t : {&ctx->cdiag_t, &ctx->cwE_t, &ctx->cwN_t})
      if (e == cudaSuccess && !*t) {
        e = dalloc(t, npad);
        if (e != cudaSuccess) *t = nullptr;
      }
    ctx->op.cdiag_t = ctx->cdiag_t;
    ctx->op.cwE_t = ctx->cwE_t;
    ctx->op.cwN_t = ctx->cwN_t;
    // the per-cell tables of the current field, now with their row-tiled copies
    if (e == cudaSuccess && ctx->op.varying)
      e = pcg::launch_column_setup(ctx->op, ctx->state, ctx->cdiag, ctx->cdiag_t, ctx->cwE_t,
                                   ctx->cwN_t, ctx->tnphi, ctx->tinvd, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "layout change");
  ctx->layout = layout;
  ctx->config_gen++;
  return PCG_OK;
}

int pcg_set_factors(pcg_ctx* ctx, int mode) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (mode != PCG_FACTORS_STORED && mode != PCG_FACTORS_RECOMPUTE)
    return fail(ctx, PCG_EINVAL, "unknown factor mode %d", mode);
  if (mode == PCG_FACTORS_RECOMPUTE && !ctx->nscratch) {
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
    const size_t count = (size_t)ctx->grid_tm * pcg::kTmWarpsPerBlock * pcg::kTile * ctx->op.nz;
    cudaError_t e = dalloc(&ctx->nscratch, count);
    if (e != cudaSuccess) {
      ctx->nscratch = nullptr;
      return cuda_fail(ctx, e, "allocation of the factor scratch");
    }
  }
  ctx->factors = mode;
  ctx->config_gen++;
  return PCG_OK;
}

// Automatic blocks per column.  Substructuring adds two fp64 operations per
// cell (the spike correction) to the six of the sweep, and on this part the
// sweep is fp64-bound as soon as the grid has a few hundred tiles of 32
// columns (measured: 128x128x64, 512 tiles, Thomas 31 us against 33 us with
// 2 or 4 blocks).  Only grids with fewer tiles than half the SMs, where the
// sweep is latency-bound, take 4 blocks (32x32x16: 14.1 us against 16.0 us),
// or fewer if the column is too short.
int auto_split(pcg_ctx* ctx) {
  if (ctx->op.ntiles * 2 >= ctx->num_sms) return 1;
  // the persistent and cluster loops (Thomas only) are faster still on these
  // grids (32x32x16: 21.8 us per iteration persistent against 24.3 us with 4
  // blocks, batched)
  if (ctx->loop_req != PCG_LOOP_BATCHED && (persistent_grid(ctx) || ctx->cl_ctas > 0)) return 1;
  for (int P = 4; P >= 2; P /= 2)
    if (pcg::split_valid(ctx->op.nz, P) && pcg::split_grid(ctx->op, P, ctx->num_sms) > 0) return P;
  return 1;
}

int pcg_set_substructuring(pcg_ctx* ctx, int nblocks) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  const int nz = ctx->op.nz;
  if (nblocks != 0 && nblocks != 1 && !pcg::split_valid(nz, nblocks))
    return fail(ctx, PCG_EINVAL,
                "nblocks %d: must be 0, 1, 2, 4, 8 or 16, with nz (%d) >= 2*nblocks-1", nblocks,
                nz);
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  int P = (nblocks == 0) ? auto_split(ctx) : nblocks;
  int grid = 0;
  if (P > 1) {
    grid = pcg::split_grid(ctx->op, P, ctx->num_sms);
    if (grid == 0)
      return fail(ctx, PCG_EINVAL, "columns of %d levels do not fit the substructured sweep", nz);
  }
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  Op& op = ctx->op;
  if (e == cudaSuccess && P != ctx->split_p) {
    double** tabs[] = {&op.sp_nphi, &op.sp_invd, &op.sp_ta,    &op.sp_tb,
                       &op.sp_corners, &op.sp_invdS, &op.sp_nphiS};
    for (double** t : tabs) {
      if (*t) cudaFree(*t);
      *t = nullptr;
    }
    ctx->split_p = 1;
    ctx->config_gen++;  // no captured sweep may keep the freed tables, even if what follows fails
    if (P > 1) {
      const size_t npad = (size_t)op.ntiles * pcg::kTile * nz;
      const size_t per_col = (size_t)op.ntiles * pcg::kTile;
      e = dalloc(&op.sp_nphi, npad);
      if (e == cudaSuccess) e = dalloc(&op.sp_invd, npad);
      if (e == cudaSuccess) e = dalloc(&op.sp_ta, npad);
      if (e == cudaSuccess) e = dalloc(&op.sp_tb, npad);
      if (e == cudaSuccess) e = dalloc(&op.sp_corners, per_col * 4 * P);
      if (e == cudaSuccess) e = dalloc(&op.sp_invdS, per_col * (P - 1));
      if (e == cudaSuccess) e = dalloc(&op.sp_nphiS, per_col * (P - 1));
    }
  }
  const size_t need = 2 * (size_t)(grid + ctx->grid_ta);
  if (e == cudaSuccess && need > ctx->partials_cap) {
    double* np = nullptr;
    e = dalloc(&np, need);
    if (e == cudaSuccess) {
      cudaFree(ctx->partials);
      ctx->partials = np;
      ctx->partials_cap = need;
    }
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "substructuring tables");
  ctx->split_req = nblocks;
  ctx->split_p = P;
  ctx->config_gen++;
  ctx->grid_sp = grid;
  return (P > 1) ? run_split_setup(ctx) : PCG_OK;
}

int pcg_set_loop(pcg_ctx* ctx, int mode) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (mode != PCG_LOOP_AUTO && mode != PCG_LOOP_BATCHED && mode != PCG_LOOP_PERSISTENT &&
      mode != PCG_LOOP_CLUSTER)
    return fail(ctx, PCG_EINVAL, "unknown loop mode %d", mode);
  ctx->loop_req = mode;
  return PCG_OK;
}

int pcg_set_preconditioner(pcg_ctx* ctx, int prec) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (prec != PCG_PREC_LINE && prec != PCG_PREC_MULTIGRID)
    return fail(ctx, PCG_EINVAL, "unknown preconditioner %d", prec);
  if (prec == ctx->prec) return PCG_OK;
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  if (prec == PCG_PREC_MULTIGRID) {
    if (ctx->layout != PCG_LAYOUT_TILED)
      return fail(ctx, PCG_EINVAL, "the multigrid preconditioner needs the row-tiled layout");
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "preconditioner change");
    int st = mg_allocate(ctx);
    if (st) return st;
    ctx->prec = prec;
    st = mg_setup(ctx);
    if (st) {
      ctx->prec = PCG_PREC_LINE;
      mg_release(ctx);
      return st;
    }
  } else {
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "preconditioner change");
    mg_release(ctx);
    ctx->prec = prec;
  }
  ctx->config_gen++;
  return PCG_OK;
}

int pcg_set_multigrid(pcg_ctx* ctx, int nu, double omega, int max_levels) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (nu < 1 || nu > 16) return fail(ctx, PCG_EINVAL, "nu must be in 1..16 (got %d)", nu);
  if (!(omega > 0.0 && omega <= 1.0))
    return fail(ctx, PCG_EINVAL, "omega must be in (0, 1] (got %g)", omega);
  if (max_levels < 0) return fail(ctx, PCG_EINVAL, "max_levels must be >= 0");
  const bool relevel = max_levels != ctx->mg_max_levels;
  if (relevel && ctx->prec == PCG_PREC_MULTIGRID &&
      mg_count_levels(ctx->op.nx, ctx->op.ny, max_levels) < 2)
    return fail(ctx, PCG_EINVAL, "multigrid needs at least two levels");
  ctx->mg_nu = nu;
  ctx->mg_omega = omega;
  ctx->mg_max_levels = max_levels;
  ctx->config_gen++;
  if (relevel && ctx->prec == PCG_PREC_MULTIGRID) {
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "multigrid change");
    int st = mg_allocate(ctx);
    if (st == PCG_OK) st = mg_setup(ctx);
    if (st) {
      ctx->prec = PCG_PREC_LINE;
      mg_release(ctx);
      return st;
    }
  }
  return PCG_OK;
}

int pcg_get_multigrid(const pcg_ctx* ctx, int* levels_out) {
  if (!ctx || !levels_out) return fail(nullptr, PCG_EINVAL, "NULL argument");
  *levels_out = ctx->prec == PCG_PREC_MULTIGRID ? (int)ctx->mg.size() + 1 : 0;
  return PCG_OK;
}

int pcg_mg_vcycle(pcg_ctx* ctx, const double* r_dev, double* z_dev) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (ctx->prec != PCG_PREC_MULTIGRID)
    return fail(ctx, PCG_EINVAL, "the multigrid preconditioner is not selected");
  if (!r_dev || !z_dev) return fail(ctx, PCG_EINVAL, "r and z must be non-NULL device pointers");
  if (overlap(r_dev, z_dev, ctx->op.n)) return fail(ctx, PCG_EINVAL, "r and z overlap");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  // the solver's own vectors serve as row-tiled scratch between solves;
  // `done` is cleared so that the cycle's kernels run
  Op op = ctx->op;
  cudaStream_t s = ctx->stream;
  cudaError_t e = cudaMemsetAsync(&ctx->state->done, 0, sizeof(int), s);
  if (e == cudaSuccess) e = pcg::launch_to_tiled(op, r_dev, ctx->p, s);
  int cnt = 0;
  if (e == cudaSuccess) e = mg_enqueue(ctx, op, ctx->p, ctx->u_t, false, s, &cnt);
  if (e == cudaSuccess) e = pcg::launch_from_tiled(op, ctx->state, ctx->u_t, nullptr, z_dev, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "multigrid V-cycle launch");
  return PCG_OK;
}

int pcg_set_az_form(pcg_ctx* ctx, int form) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (form != PCG_AZ_AUTO && form != PCG_AZ_STENCIL && form != PCG_AZ_RESIDUAL)
    return fail(ctx, PCG_EINVAL, "unknown form of A z %d", form);
  if (form != ctx->az_req) ctx->config_gen++;  // the captured sweeps change
  ctx->az_req = form;
  return PCG_OK;
}

int pcg_get_az_form(const pcg_ctx* ctx, int* form_out) {
  if (!ctx || !form_out) return fail(nullptr, PCG_EINVAL, "NULL argument");
  *form_out = resolved_az(ctx);
  return PCG_OK;
}

int pcg_test_tensor_memory(pcg_ctx* ctx, int enable) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  ctx->tmem_off = enable == 0;
  return PCG_OK;
}

int pcg_test_poison_work(pcg_ctx* ctx) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  // every byte 0xFF: each double is a NaN, padding included
  const size_t bytes = sizeof(double) * (size_t)(ctx->op.ntiles * pcg::kTile * ctx->op.nz);
  cudaError_t e = cudaSuccess;
  for (double* v : {ctx->r, ctx->z, ctx->p, ctx->q, ctx->u_t})
    if (v && e == cudaSuccess) e = cudaMemsetAsync(v, 0xFF, bytes, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "work vector fill");
  return PCG_OK;
}

int pcg_test_barrier_absent(pcg_ctx* ctx, int absent) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (absent < 0) return fail(ctx, PCG_EINVAL, "absent must be >= 0");
  ctx->test_absent = (unsigned int)absent;
  return PCG_OK;
}

int pcg_get_loop(const pcg_ctx* ctx, int* mode_out) {
  if (!ctx || !mode_out) return fail(nullptr, PCG_EINVAL, "NULL argument");
  *mode_out = resolved_loop(ctx);
  return PCG_OK;
}

int pcg_get_substructuring(const pcg_ctx* ctx, int* nblocks_out) {
  if (!ctx || !nblocks_out) return fail(nullptr, PCG_EINVAL, "NULL argument");
  *nblocks_out = ctx->split_p;
  return PCG_OK;
}

int pcg_set_stream(pcg_ctx* ctx, void* stream) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  cudaStream_t next = static_cast<cudaStream_t>(stream);
  if (next != ctx->stream) {
    // work queued on the old stream (a coefficient upload, a standalone
    // operator) comes before the new stream's
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
    cudaEvent_t ev = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(next, ev, 0);
    if (ev) cudaEventDestroy(ev);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "stream switch");
  }
  ctx->stream = next;
  return PCG_OK;
}

int pcg_apply_A(pcg_ctx* ctx, const double* x_dev, double* y_dev) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (!x_dev || !y_dev) return fail(ctx, PCG_EINVAL, "x and y must be non-NULL device pointers");
  if (overlap(x_dev, y_dev, ctx->op.n)) return fail(ctx, PCG_EINVAL, "x and y overlap");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e = pcg::launch_apply(ctx->op, x_dev, y_dev, ctx->grid_a, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "apply_A launch");
  return PCG_OK;
}

int pcg_precond(pcg_ctx* ctx, const double* r_dev, double* z_dev) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (!r_dev || !z_dev) return fail(ctx, PCG_EINVAL, "r and z must be non-NULL device pointers");
  if (overlap(r_dev, z_dev, ctx->op.n)) return fail(ctx, PCG_EINVAL, "r and z overlap");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e =
      (ctx->tmem_ok && !ctx->tmem_off && pcg::precond_tmem_supported(ctx->op, r_dev, nullptr, z_dev))
          ? pcg::launch_precond_tmem(ctx->op, ctx->state, const_cast<double*>(r_dev), nullptr,
                                     z_dev, nullptr, nullptr, false,
                                     pcg::grid_precond_tmem(ctx->op, ctx->num_sms), ctx->stream)
          : pcg::launch_precond(ctx->op, ctx->state, r_dev, z_dev, ctx->grid_m, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "precond launch");
  return PCG_OK;
}

static int check_solve_args(pcg_ctx* ctx, const double* b, const double* x, double rtol,
                            int maxit) {
  if (!b || !x) return fail(ctx, PCG_EINVAL, "b and x must be non-NULL");
  if (!(std::isfinite(rtol) && rtol >= 0.0)) return fail(ctx, PCG_EINVAL, "rtol must be >= 0");
  if (maxit < 0) return fail(ctx, PCG_EINVAL, "maxit must be >= 0");
  if (overlap(b, x, ctx->op.n)) return fail(ctx, PCG_EINVAL, "b and x overlap");
  return PCG_OK;
}

int pcg_solve(pcg_ctx* ctx, const double* b_dev, double* x_dev, double rtol, int maxit,
              int* iters_out, double* res_hist) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  int st = check_solve_args(ctx, b_dev, x_dev, rtol, maxit);
  if (st) return st;
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  return solve_device(ctx, b_dev, x_dev, rtol, maxit, iters_out, res_hist);
}

int pcg_solve_from_zero(pcg_ctx* ctx, const double* b_dev, double* x_dev, double rtol,
                        int maxit, int* iters_out, double* res_hist) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  int st = check_solve_args(ctx, b_dev, x_dev, rtol, maxit);
  if (st) return st;
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  if (ctx->layout == PCG_LAYOUT_TILED) {
    ctx->x0_zero = true;  // the row-tiled start is told; x is written, never read
  } else {
    const cudaError_t e =
        cudaMemsetAsync(x_dev, 0, sizeof(double) * (size_t)ctx->op.n, ctx->stream);  // +0.0
    if (e != cudaSuccess) return cuda_fail(ctx, e, "initial guess");
  }
  return solve_device(ctx, b_dev, x_dev, rtol, maxit, iters_out, res_hist);
}

// Device copies of b and x for the host-buffer entry points (made on first use).
static cudaError_t host_api_buffers(pcg_ctx* ctx) {
  cudaError_t e = cudaSuccess;
  if (!ctx->b_host_api) e = dalloc(&ctx->b_host_api, ctx->op.n);
  if (e == cudaSuccess && !ctx->x_host_api) e = dalloc(&ctx->x_host_api, ctx->op.n);
  return e;
}

// The copy-outs of earlier asynchronous calls, finished (host side).
static cudaError_t wait_copy_outs(pcg_ctx* ctx) {
  if (!ctx->out_stream) return cudaSuccess;
  cudaError_t e = cudaStreamSynchronize(ctx->out_stream);
  if (e == cudaSuccess) ctx->out_pending[0] = ctx->out_pending[1] = false;
  return e;
}

static int check_host_x0(pcg_ctx* ctx, const double* b_host, const double* x0_host,
                         const double* x_host) {
  if (x0_host && x0_host != x_host && overlap(b_host, x0_host, ctx->op.n))
    return fail(ctx, PCG_EINVAL, "b and x0 overlap");
  return PCG_OK;
}

// A zero initial guess (x0_host NULL) is set on the device only where the
// solve reads it: the column layout's start does, the row-tiled start is told
// instead (pcg_ctx::x0_zero).
static bool zero_x0_skips_copy(const pcg_ctx* ctx, const double* x0_host) {
  return !x0_host && ctx->layout == PCG_LAYOUT_TILED;
}

// Solve from the device copies, then copy x out and wait for it.
static int solve_copy_out(pcg_ctx* ctx, bool x0_zero, double* x_host, double rtol, int maxit,
                          int* iters_out, double* res_hist) {
  ctx->x0_zero = x0_zero;
  int st = solve_device(ctx, ctx->b_host_api, ctx->x_host_api, rtol, maxit, iters_out, res_hist);
  if (st != PCG_OK && st != PCG_ENOTCONV && st != PCG_EBREAKDOWN) return st;
  const size_t bytes = sizeof(double) * (size_t)ctx->op.n;
  cudaError_t e =
      cudaMemcpyAsync(x_host, ctx->x_host_api, bytes, cudaMemcpyDeviceToHost, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy");
  return st;
}

int pcg_solve_host_x0(pcg_ctx* ctx, const double* b_host, const double* x0_host, double* x_host,
                      double rtol, int maxit, int* iters_out, double* res_hist) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  int st = check_solve_args(ctx, b_host, x_host, rtol, maxit);
  if (!st) st = check_host_x0(ctx, b_host, x0_host, x_host);
  if (st) return st;
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e = wait_copy_outs(ctx);  // an asynchronous call's copy-out may read x_host_api
  if (e == cudaSuccess) e = host_api_buffers(ctx);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device buffers for b and x");
  const size_t bytes = sizeof(double) * (size_t)ctx->op.n;
  const bool x0_zero = zero_x0_skips_copy(ctx, x0_host);
  e = cudaMemcpyAsync(ctx->b_host_api, b_host, bytes, cudaMemcpyHostToDevice, ctx->stream);
  if (e == cudaSuccess && x0_host)
    e = cudaMemcpyAsync(ctx->x_host_api, x0_host, bytes, cudaMemcpyHostToDevice, ctx->stream);
  if (e == cudaSuccess && !x0_host && !x0_zero)
    e = cudaMemsetAsync(ctx->x_host_api, 0, bytes, ctx->stream);  // x0 = +0.0
  if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
  return solve_copy_out(ctx, x0_zero, x_host, rtol, maxit, iters_out, res_hist);
}

// pcg_update_solve_host (async false) and pcg_update_solve_host_async.
static int update_solve_host(pcg_ctx* ctx, const pcg_coeffs* coeffs, const double* b_host,
                             const double* x0_host, double* x_host, double rtol, int maxit,
                             int* iters_out, double* res_hist, bool async) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  int st = validate_coeffs(ctx, ctx->op.nx, ctx->op.ny, ctx->op.nz, coeffs, true);
  if (st) return st;
  const bool varying = coeffs->a_h_field != nullptr;
  if (varying && !ctx->has_field_buffers)
    return fail(ctx, PCG_EINVAL,
                "context was created with a constant a_h; it cannot take an a_h field");
  st = check_solve_args(ctx, b_host, x_host, rtol, maxit);
  if (!st) st = check_host_x0(ctx, b_host, x0_host, x_host);
  if (st) return st;
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e = async ? cudaSuccess : wait_copy_outs(ctx);
  if (e == cudaSuccess) e = host_api_buffers(ctx);
  if (e == cudaSuccess && !ctx->copy_stream)
    e = cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess && !ctx->copy_done)
    e = cudaEventCreateWithFlags(&ctx->copy_done, cudaEventDisableTiming);
  if (async) {
    if (e == cudaSuccess && !ctx->x_async2) e = dalloc(&ctx->x_async2, ctx->op.n);
    if (e == cudaSuccess && !ctx->out_stream)
      e = cudaStreamCreateWithFlags(&ctx->out_stream, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&ctx->out_done[0], &ctx->out_done[1], &ctx->solved})
      if (e == cudaSuccess && !*ev) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  }
  // no earlier work on the context's stream may still use the device copies
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device buffers for b and x");
  // the device copy of x: the asynchronous calls alternate between two, so
  // that one call's copy-out overlaps the next call's solve; a copy-out still
  // reading the one used now is waited for on the device, by both streams
  // that write it (x0 in, the solve)
  const int slot = async ? ctx->out_slot : 0;
  double* xs = slot ? ctx->x_async2 : ctx->x_host_api;
  if (async && ctx->out_pending[slot]) {
    e = cudaStreamWaitEvent(ctx->copy_stream, ctx->out_done[slot], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->stream, ctx->out_done[slot], 0);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy order");
  }
  // b or x0 in a host buffer that an earlier call's copy-out may still be
  // writing (a sequence of solves each started from the last solution): the
  // copy-in waits for that copy-out on the device
  for (int k = 0; k < 2 && async; ++k) {
    const long long n = ctx->op.n;
    if (ctx->out_pending[k] && (overlap(b_host, n, ctx->out_host[k], n) ||
                                (x0_host && overlap(x0_host, n, ctx->out_host[k], n)))) {
      e = cudaStreamWaitEvent(ctx->copy_stream, ctx->out_done[k], 0);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy order");
    }
  }
  const size_t bytes = sizeof(double) * (size_t)ctx->op.n;
  const bool x0_zero = zero_x0_skips_copy(ctx, x0_host);
  bool copies_enqueued = false;
  auto copy_in = [&]() -> cudaError_t {
    copies_enqueued = true;
    cudaError_t ce = cudaMemcpyAsync(ctx->b_host_api, b_host, bytes, cudaMemcpyHostToDevice,
                                     ctx->copy_stream);
    if (ce == cudaSuccess && x0_host)
      ce = cudaMemcpyAsync(xs, x0_host, bytes, cudaMemcpyHostToDevice, ctx->copy_stream);
    if (ce == cudaSuccess && !x0_host && !x0_zero)
      ce = cudaMemsetAsync(xs, 0, bytes, ctx->copy_stream);  // x0 = +0.0
    if (ce == cudaSuccess) ce = cudaEventRecord(ctx->copy_done, ctx->copy_stream);
    return ce;
  };
  st = load_coeffs(ctx, coeffs, varying, copy_in);
  if (st) {
    if (copies_enqueued) cudaStreamSynchronize(ctx->copy_stream);
    return st;
  }
  e = cudaStreamWaitEvent(ctx->stream, ctx->copy_done, 0);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
  if (!async) return solve_copy_out(ctx, x0_zero, x_host, rtol, maxit, iters_out, res_hist);
  // asynchronous: the solve, then x out on out_stream, not waited for
  ctx->x0_zero = x0_zero;
  st = solve_device(ctx, ctx->b_host_api, xs, rtol, maxit, iters_out, res_hist);
  if (st != PCG_OK && st != PCG_ENOTCONV && st != PCG_EBREAKDOWN) return st;
  e = cudaEventRecord(ctx->solved, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->out_stream, ctx->solved, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(x_host, xs, bytes, cudaMemcpyDeviceToHost, ctx->out_stream);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->out_done[slot], ctx->out_stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy");
  ctx->out_pending[slot] = true;
  ctx->out_host[slot] = x_host;
  ctx->out_slot = slot ^ 1;
  return st;
}

int pcg_update_solve_host(pcg_ctx* ctx, const pcg_coeffs* coeffs, const double* b_host,
                          const double* x0_host, double* x_host, double rtol, int maxit,
                          int* iters_out, double* res_hist) {
  return update_solve_host(ctx, coeffs, b_host, x0_host, x_host, rtol, maxit, iters_out,
                           res_hist, false);
}

int pcg_update_solve_host_async(pcg_ctx* ctx, const pcg_coeffs* coeffs, const double* b_host,
                                const double* x0_host, double* x_host, double rtol, int maxit,
                                int* iters_out, double* res_hist) {
  return update_solve_host(ctx, coeffs, b_host, x0_host, x_host, rtol, maxit, iters_out,
                           res_hist, true);
}

int pcg_host_wait(pcg_ctx* ctx) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  const cudaError_t e = wait_copy_outs(ctx);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy");
  return PCG_OK;
}

int pcg_solve_host(pcg_ctx* ctx, const double* b_host, double* x_host, double rtol, int maxit,
                   int* iters_out, double* res_hist) {
  return pcg_solve_host_x0(ctx, b_host, x_host, x_host, rtol, maxit, iters_out, res_hist);
}

int pcg_precond_dot_noalloc(pcg_ctx* ctx, const double* r_dev, double* z_dev, double* rz_dev) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  if (!r_dev || !z_dev || !rz_dev)
    return fail(ctx, PCG_EINVAL, "r, z and rz must be non-NULL device pointers");
  if (overlap(r_dev, z_dev, ctx->op.n)) return fail(ctx, PCG_EINVAL, "r and z overlap");
  // rz is one value: only an rz inside r or z overlaps them
  if (overlap(rz_dev, 1, r_dev, ctx->op.n) || overlap(rz_dev, 1, z_dev, ctx->op.n))
    return fail(ctx, PCG_EINVAL, "rz overlaps r or z");
  if (ctx->op.ntiles > pcg::kNoallocMaxTiles)
    return fail(ctx, PCG_EINVAL,
                "grid has %lld columns; the no-allocation scratch holds at most %lld "
                "(%lld tiles of 32 columns)",
                ctx->op.ncols, pcg::kNoallocMaxTiles * pcg::kTile, pcg::kNoallocMaxTiles);
  DeviceGuard g(ctx->device);
  if (!g.ok) return fail(ctx, PCG_ECUDA, "cannot make device %d current", ctx->device);
  cudaError_t e = pcg::launch_precond_dot_noalloc(ctx->op, r_dev, z_dev, rz_dev,
                                                  ctx->noalloc_partials, ctx->num_sms,
                                                  ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "precond_dot_noalloc");
  return PCG_OK;
}

int pcg_measure_fp64_rate(int warps_per_sm, int launches, double* lane_ops_per_s,
                          double* sm_mhz, double* lanes_per_sm_clk) {
  if (warps_per_sm < 1 || warps_per_sm > 64 || (warps_per_sm > 4 && warps_per_sm % 4 != 0))
    return fail(nullptr, PCG_EINVAL,
                "warps_per_sm must be 1, 2, 3 or a multiple of 4 in [4, 64]");
  if (launches < 1 || launches > 100)
    return fail(nullptr, PCG_EINVAL, "launches must be in [1, 100]");
  if (!lane_ops_per_s || !sm_mhz || !lanes_per_sm_clk)
    return fail(nullptr, PCG_EINVAL, "NULL output pointer");
  int dev = 0, nsm = 0, clk_khz = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "device query");
  // four warps per block, one per sub-partition; below four warps per SM, one
  // block per SM with warps on sub-partitions 0 .. warps_per_sm-1
  const int threads = 32 * std::min(warps_per_sm, 4);
  const int blocks = nsm * std::max(warps_per_sm / 4, 1);
  // about 20 ms per launch at 2 lane operations per SM per clock
  const double per_trip = (double)pcg::fp64_rate_lane_ops(blocks, threads, 1);
  const int trips = std::max(1, (int)(0.02 * 2.0 * nsm * clk_khz * 1e3 / per_trip));
  double* sink = nullptr;
  unsigned long long* stamps = nullptr;
  cudaStream_t s = nullptr;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  e = cudaMalloc(&sink, sizeof(double) * blocks);
  if (e == cudaSuccess) e = cudaMalloc(&stamps, sizeof(unsigned long long) * 2 * blocks);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreate(&ev[0]);
  if (e == cudaSuccess) e = cudaEventCreate(&ev[1]);
  std::vector<unsigned long long> st(2 * (size_t)blocks);
  double best = 0.0, best_mhz = 0.0;
  for (int l = -1; e == cudaSuccess && l < launches; ++l) {  // l = -1: warm-up
    e = cudaEventRecord(ev[0], s);
    if (e == cudaSuccess) e = pcg::launch_fp64_rate(blocks, threads, trips, sink, stamps, s);
    if (e == cudaSuccess) e = cudaEventRecord(ev[1], s);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev[1]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
    if (e == cudaSuccess)
      e = cudaMemcpy(st.data(), stamps, sizeof(unsigned long long) * st.size(),
                     cudaMemcpyDeviceToHost);
    if (e != cudaSuccess || l < 0 || ms <= 0.f) continue;
    std::vector<double> mhz;
    mhz.reserve(blocks);
    for (int b = 0; b < blocks; ++b)
      if (st[2 * b + 1] > 0) mhz.push_back(1e3 * (double)st[2 * b] / (double)st[2 * b + 1]);
    std::sort(mhz.begin(), mhz.end());
    const double rate = (double)pcg::fp64_rate_lane_ops(blocks, threads, trips) / (ms * 1e-3);
    if (rate > best) {
      best = rate;
      best_mhz = mhz.empty() ? 0.0 : mhz[mhz.size() / 2];
    }
  }
  if (ev[1]) cudaEventDestroy(ev[1]);
  if (ev[0]) cudaEventDestroy(ev[0]);
  if (s) cudaStreamDestroy(s);
  if (stamps) cudaFree(stamps);
  if (sink) cudaFree(sink);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "fp64 rate probe");
  *lane_ops_per_s = best;
  *sm_mhz = best_mhz;
  *lanes_per_sm_clk = best_mhz > 0.0 ? best / (nsm * best_mhz * 1e6) : 0.0;
  return PCG_OK;
}

const char* pcg_last_error(const pcg_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

int pcg_enable_timing(pcg_ctx* ctx, int enable) {
  if (!ctx) return fail(nullptr, PCG_EINVAL, "ctx is NULL");
  ctx->timing = enable != 0;
  for (int i = 0; i < PCG_K_COUNT; ++i) {
    ctx->ms[i] = 0.0;
    ctx->launches[i] = 0;
  }
  return PCG_OK;
}

int pcg_kernel_times(pcg_ctx* ctx, double* ms_out, long long* launches_out) {
  if (!ctx || !ms_out || !launches_out) return fail(ctx, PCG_EINVAL, "NULL argument");
  for (int i = 0; i < PCG_K_COUNT; ++i) {
    ms_out[i] = ctx->ms[i];
    launches_out[i] = ctx->launches[i];
  }
  return PCG_OK;
}

int pcg_launch_info(const pcg_ctx* ctx, int* grid_precond, int* grid_spmv,
                    long long* last_solve_launches) {
  if (!ctx) return PCG_EINVAL;
  const bool tiled = ctx->layout == PCG_LAYOUT_TILED;
  if (grid_precond)
    *grid_precond = tiled ? (ctx->split_p > 1 ? ctx->grid_sp : ctx->grid_tm) : ctx->grid_m;
  if (grid_spmv) *grid_spmv = tiled ? ctx->grid_ta : ctx->grid_a;
  if (last_solve_launches) *last_solve_launches = ctx->last_launches;
  return PCG_OK;
}

}  // extern "C"
