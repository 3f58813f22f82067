// sla_cg_solve_static: the CG solve for callers that cannot allocate device memory.
//
// Some callers can neither call cudaMalloc nor hand the library a workspace: plugins
// loaded into a host application that owns and budgets every byte of device memory,
// code on latency-critical paths where an allocation (and the device synchronisation
// it can imply) is not allowed, and thin bindings that have no device allocator at
// all.  For them this entry point keeps its scratch in a fixed array in the library's
// own device memory.  The array is reserved on a GPU when this file's device code is
// loaded there, which (under CUDA's lazy module loading) is the first call on that GPU,
// and it is held until the process exits.  The caller still passes the matrix, b, x0
// and x.
//
// Limits: one system (no batch) of at most kStaticMaxN = 65,536 unknowns, fp32 or fp64,
// with or without Jacobi; larger systems are rejected with SLA_WORKSPACE_TOO_SMALL
// before anything is launched.  The iteration runs the same kernels as sla_cg_solve,
// driven from the host (no graph is instantiated, since that may allocate).
#include <cuda_runtime.h>

#include <mutex>

#include "sla_common.cuh"
#include "sla_host.h"

namespace sla {

namespace {

constexpr int64_t kStaticMaxN = 65536;
// The workspace layout of the largest case: n = 65,536, one system, fp64 values, Jacobi, no row
// bitmap (the host-driven loop never runs the resident kernel): Glob (256 B) + Ctl (256 B) +
// partial sums (6 x 2048 doubles = 98,304 B) + 6 vectors of 65,536 doubles (524,288 B each:
// r, p0, p1, q, 1/diag, z).  Every smaller or fp32 case needs less.
constexpr size_t kStaticScratchBytes = make_layout(kStaticMaxN, 1, sizeof(double), true, false).total;
static_assert(kStaticScratchBytes == 3244544, "the documented size of the static scratch");
constexpr int kMaxDevices = 64;

// The shared scratch.  In host code this name is only a stand-in for the device symbol:
// never pass it to a kernel; use the address returned by cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device (with that
// device current) and cached.
sla_status static_scratch(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e);
  if (dev < 0 || dev >= kMaxDevices) return SLA_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return fail(e);
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return SLA_OK;
}

}  // namespace

}  // namespace sla

using namespace sla;

extern "C" SLA_API sla_status sla_cg_solve_static(const sla_csr *A, const void *b, const void *x0,
                                                  const sla_cg_opts *opts, void *x, sla_cg_info *info,
                                                  double *history, void *stream) {
  // argument checks first (the same as sla_cg_solve's): they need no GPU
  SLA_CHECK(check_csr(A, true));
  SLA_CHECK(check_vec(b, A, false));
  SLA_CHECK(check_vec(x0, A, true));
  SLA_CHECK(check_vec(x, A, false));
  if (!aligned(history, 8)) return SLA_INVALID_ARG;
  if (!opts) return SLA_INVALID_ARG;
  sla_cg_opts o = *opts;
  o.loop = SLA_LOOP_HOST;  // the only loop that needs no graph (instantiating one may allocate)
  SLA_CHECK(check_opts(&o));
  if (A->n > kStaticMaxN) return SLA_WORKSPACE_TOO_SMALL;  // beyond the static scratch
  const size_t vsz = A->dtype == SLA_F64 ? 8 : 4;
  const bool jac = opts->precond == SLA_PRECOND_JACOBI;
  const Layout L = make_layout(A->n, 1, vsz, jac, /*with_halo=*/false);  // the host loop needs no row bitmap
  if (L.total > kStaticScratchBytes) return SLA_WORKSPACE_TOO_SMALL;
  if (A->n == 0) {
    if (info) {
      info->iters = 0;
      info->rel_res = 0.0;
      info->status = SLA_OK;
      info->path = 0;
      info->kernels = 0;
    }
    return SLA_OK;
  }
  void *ws = nullptr;
  sla_status s = static_scratch(&ws);
  if (s != SLA_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  // The init kernel of the solve zeroes the control block and the loop state in the scratch, so
  // nothing left by an earlier call is read; vectors are written before they are read.
  s = cg_entry(A, 1, A->values, 0, b, x0, &o, x, nullptr, history, ws, st, /*halo_ws=*/false);
  if (s != SLA_OK || !info) return s;
  Ctl hc;
  Glob hg;
  cudaError_t e = cudaMemcpyAsync(&hc, (const char *)ws + L.ctl, sizeof(Ctl), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hg, (const char *)ws + L.glob, sizeof(Glob), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(e);
  count_launches(hg.kernels);
  info->iters = hc.k;
  info->rel_res = hc.rel_res;
  info->status = hg.bad_csr ? SLA_BAD_CSR : hc.status;
  info->path = SLA_LOOP_HOST;
  info->kernels = (int64_t)hg.kernels;
  return SLA_OK;
}
