// libsla C ABI: argument checks, SpMV, the sparse-pattern gradient, CSR validation,
// and the solve / adjoint entry points (which run the device-resident CG of sla_cg.cu).
//
// Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers
// and Sparse Tensor Parallelism for PyTorch" (Chi, Wen), technical summary,
// Methodology 1 (.matvec / .solve over one matrix or a shared-pattern batch)
// and Methodology 2 (linear adjoint: grad_b = lambda, grad_A = -lambda_i x_j on
// the sparsity pattern).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "sla_common.cuh"
#include "sla_host.h"
#include "sla_pattern.cuh"

namespace sla {

namespace {
thread_local cudaError_t t_last_error = cudaSuccess;
std::atomic<uint64_t> g_launches{0};
}  // namespace

sla_status fail(cudaError_t e) {
  t_last_error = e;
  return SLA_CUDA_ERROR;
}

void count_launches(uint64_t k) { g_launches.fetch_add(k); }

namespace {
thread_local int t_last_path = 0;
}
void set_last_path(int path) { t_last_path = path; }

sla_status read_info(const Ctl *ctl, const Glob *glob, int64_t batch, cudaStream_t stream, sla_cg_info *info) {
  std::vector<Ctl> hc((size_t)batch);
  Glob hg;
  cudaError_t e = cudaMemcpyAsync(hc.data(), ctl, sizeof(Ctl) * (size_t)batch, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hg, glob, sizeof(Glob), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(e);
  count_launches(hg.kernels);
  for (int64_t s = 0; s < batch; ++s) {
    info[s].iters = hc[s].k;
    info[s].rel_res = hc[s].rel_res;
    info[s].status = hg.bad_csr ? SLA_BAD_CSR : hc[s].status;
    info[s].path = t_last_path;
    info[s].kernels = (int64_t)hg.kernels;
  }
  return SLA_OK;
}

// ------------------------------------------------------------------------ kernels

// y = A x, one thread per row, row sums in storage order with fused multiply-adds.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) spmv_kernel(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                      const int32_t *__restrict__ ci, const V *__restrict__ val,
                                                      const V *__restrict__ x, V *__restrict__ y) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, i, nnz, e0, e1, nullptr);
    V acc = V(0);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t c = ci[e];
      if (col_ok(c, (int32_t)n, nullptr)) acc = fmav<V>(val[e], x[c], acc);
    }
    y[i] = acc;
  }
}

// gv[s][k] = -lambda_s[row(k)] * x_s[col(k)]: one streaming pass over the pattern (sla_pattern.cuh),
// lambda staged per row tile in shared memory, x gathered per entry; blockIdx.y = system.
template <typename V, typename I>
__global__ void __launch_bounds__(kPatBlock, kPatMinBlocks) grad_values_kernel(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                                const int32_t *__restrict__ ci,
                                                                const V *__restrict__ lam, const V *__restrict__ x,
                                                                V *__restrict__ gv) {
  __shared__ PatSmem<V> sm;
  const int s = blockIdx.y;
  lam += (int64_t)s * n;
  x += (int64_t)s * n;
  gv += (int64_t)s * nnz;
  pattern_pass<V, I>(
      n, nnz, rp, ci, sm, [&](int64_t i) { return __ldcs(lam + i); }, [](V l) { return l; },
      [&](int32_t c) { return __ldg(x + c); },
      [&](int64_t e, int64_t, V li, int32_t c, V xc) {
        __stcs(gv + e, (uint32_t)c < (uint32_t)n ? -(li * xc) : V(0));
      });
}

// gv[e] = gy[row(e)] * x[col(e)]: the gradient of L(A x) with respect to the stored values, for
// gy = dL/dy (one rounded product per entry), by the same streaming pass.
template <typename V, typename I>
__global__ void __launch_bounds__(kPatBlock, kPatMinBlocks) matvec_grad_kernel(int64_t n, int64_t nnz,
                                                                               const I *__restrict__ rp,
                                                                               const int32_t *__restrict__ ci,
                                                                               const V *__restrict__ gy,
                                                                               const V *__restrict__ x,
                                                                               V *__restrict__ gv) {
  __shared__ PatSmem<V> sm;
  pattern_pass<V, I>(
      n, nnz, rp, ci, sm, [&](int64_t i) { return __ldcs(gy + i); }, [](V a) { return a; },
      [&](int32_t c) { return __ldg(x + c); },
      [&](int64_t e, int64_t, V gi, int32_t c, V xc) {
        __stcs(gv + e, (uint32_t)c < (uint32_t)n ? gi * xc : V(0));
      });
}

// y = A^T x for a structurally symmetric pattern (every stored (j, i) has a stored (i, j)): row j
// gathers a_ij x_i over the columns i of its own row, in their (increasing) order, each a_ij found
// by a binary search in row i.  One thread per row; deterministic.  A missing partner entry is
// skipped and raises *bad (when given).
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) spmv_t_kernel(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                        const int32_t *__restrict__ ci,
                                                        const V *__restrict__ val, const V *__restrict__ x,
                                                        V *__restrict__ y, uint32_t *bad) {
  for (int64_t j = blockIdx.x * (int64_t)kBlock + threadIdx.x; j < n; j += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, j, nnz, e0, e1, bad);
    V acc = V(0);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t i = ci[e];
      if (!col_ok(i, (int32_t)n, bad)) continue;
      int64_t lo, hi;
      row_range(rp, i, nnz, lo, hi, bad);
      --hi;
      bool found = false;
      while (lo <= hi) {
        const int64_t mid = (lo + hi) >> 1;
        const int32_t cm = ci[mid];
        if (cm == (int32_t)j) {
          acc = fmav<V>(val[mid], x[i], acc);
          found = true;
          break;
        }
        if (cm < (int32_t)j) lo = mid + 1;
        else hi = mid - 1;
      }
      if (!found && bad) atomicOr(bad, 1u);
    }
    y[j] = acc;
  }
}

// Structural CSR check; records the smallest offending row.
template <typename I>
__global__ void __launch_bounds__(kBlock) validate_kernel(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                          const int32_t *__restrict__ ci, const void *values,
                                                          int dtype, int check_sym,
                                                          unsigned long long *bad_row) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    bool ok = true;
    const int64_t e0 = rp[i], e1 = rp[i + 1];
    if (i == 0 && e0 != 0) ok = false;
    if (i == n - 1 && e1 != nnz) ok = false;
    if (e1 < e0 || e0 < 0 || e1 > nnz) ok = false;
    bool diag = false;
    if (ok) {
      int64_t prev = -1;
      for (int64_t e = e0; e < e1; ++e) {
        const int64_t c = ci[e];
        if (c <= prev || c < 0 || c >= n) { ok = false; break; }
        if (c == i) diag = true;
        prev = c;
        if (check_sym) {
          // find (c, i) in row c (only within a well-formed row range)
          int64_t lo = rp[c], hi = rp[c + 1] - 1;
          if (lo < 0 || hi + 1 < lo || hi + 1 > nnz) { ok = false; break; }
          bool found = false;
          while (lo <= hi) {
            const int64_t mid = (lo + hi) >> 1;
            const int32_t cm = ci[mid];
            if (cm == i) { found = true; lo = mid; break; }
            if (cm < i) lo = mid + 1; else hi = mid - 1;
          }
          if (!found) { ok = false; break; }
          if (dtype == SLA_F64) {
            const unsigned long long a = ((const unsigned long long *)values)[e];
            const unsigned long long b = ((const unsigned long long *)values)[lo];
            if (a != b) { ok = false; break; }
          } else {
            const unsigned a = ((const unsigned *)values)[e], b = ((const unsigned *)values)[lo];
            if (a != b) { ok = false; break; }
          }
        }
      }
    }
    if (!diag) ok = false;
    if (!ok) atomicMin(bad_row, (unsigned long long)i);
  }
}

// ------------------------------------------------------------------------ helpers

namespace {

// Blocks of a pattern pass: one per row tile, at most as many as are resident on the device at once
// (the remaining tiles are taken round-robin).
int pattern_grid(int64_t n) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (n + kPatRows - 1) / kPatRows;
  const int64_t cap = (int64_t)sms * kPatMinBlocks;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

int grid_for(int64_t work, int per_block_rows) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (work + per_block_rows - 1) / per_block_rows;
  int64_t cap = (int64_t)sms * 16;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

}  // namespace

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

sla_status check_csr(const sla_csr *A, bool need_values) {
  if (!A) return SLA_INVALID_ARG;
  if (A->n < 0 || A->nnz < 0 || A->n >= ((int64_t)1 << 31)) return SLA_INVALID_ARG;
  if (A->dtype != SLA_F32 && A->dtype != SLA_F64) return SLA_INVALID_ARG;
  if (A->rowptr_type != SLA_I32 && A->rowptr_type != SLA_I64) return SLA_INVALID_ARG;
  if (A->rowptr_type == SLA_I32 && A->nnz >= ((int64_t)1 << 31)) return SLA_INVALID_ARG;
  if (A->n > 0 && !A->row_ptr) return SLA_INVALID_ARG;
  if (A->nnz > 0 && !A->col_idx) return SLA_INVALID_ARG;
  if (need_values && A->nnz > 0 && !A->values) return SLA_INVALID_ARG;
  const size_t isz = A->rowptr_type == SLA_I64 ? 8 : 4, vsz = A->dtype == SLA_F64 ? 8 : 4;
  if (!aligned(A->row_ptr, isz) || !aligned(A->col_idx, 4) || (need_values && !aligned(A->values, vsz)))
    return SLA_INVALID_ARG;
  return SLA_OK;
}

sla_status check_vec(const void *p, const sla_csr *A, bool allow_null) {
  if (!p) return (allow_null || A->n == 0) ? SLA_OK : SLA_INVALID_ARG;
  return aligned(p, A->dtype == SLA_F64 ? 8 : 4) ? SLA_OK : SLA_INVALID_ARG;
}

sla_status check_opts(const sla_cg_opts *o) {
  if (!o) return SLA_INVALID_ARG;
  if (!(o->rtol >= 0.0) || !std::isfinite(o->rtol)) return SLA_INVALID_ARG;
  if (o->maxit < 0 || o->maxit > ((int64_t)1 << 40)) return SLA_INVALID_ARG;
  if (o->precond != SLA_PRECOND_NONE && o->precond != SLA_PRECOND_JACOBI) return SLA_INVALID_ARG;
  if (o->unroll < 0 || o->unroll > 64) return SLA_INVALID_ARG;
  if (o->loop < SLA_LOOP_AUTO || o->loop > SLA_LOOP_CLUSTER) return SLA_INVALID_ARG;
  if (o->reserved != 0) return SLA_INVALID_ARG;
  return SLA_OK;
}

namespace {

sla_status check_ws(const sla_csr *A, int64_t batch, const sla_cg_opts *o, void *ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, 256)) return SLA_INVALID_ARG;
  if (ws_bytes < workspace_bytes(A->n, batch, A->dtype, o->precond)) return SLA_WORKSPACE_TOO_SMALL;
  return SLA_OK;
}

void fill_empty(sla_cg_info *info, int64_t batch) {
  if (!info) return;
  for (int64_t s = 0; s < batch; ++s) {
    info[s].iters = 0;
    info[s].rel_res = 0.0;
    info[s].status = SLA_OK;
    info[s].path = 0;
    info[s].kernels = 0;
  }
}

template <typename V, typename I>
void launch_spmv(const sla_csr *A, const void *x, void *y, cudaStream_t st) {
  spmv_kernel<V, I><<<grid_for(A->n, kBlock * 4), kBlock, 0, st>>>(A->n, A->nnz, (const I *)A->row_ptr,
                                                                   A->col_idx, (const V *)A->values, (const V *)x,
                                                                   (V *)y);
}

template <typename V, typename I>
void launch_grad(const sla_csr *A, int64_t batch, const void *lam, const void *x, void *gv, cudaStream_t st) {
  dim3 grid(pattern_grid(A->n), (unsigned)batch);
  grad_values_kernel<V, I><<<grid, kPatBlock, 0, st>>>(A->n, A->nnz, (const I *)A->row_ptr, A->col_idx,
                                                    (const V *)lam, (const V *)x, (V *)gv);
}

}  // namespace

sla_status grad_values_entry(const sla_csr *A, int64_t batch, const void *lam, const void *x, void *gv,
                             cudaStream_t st) {
  if (A->n == 0 || batch == 0) return SLA_OK;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) launch_grad<double, int64_t>(A, batch, lam, x, gv, st);
    else launch_grad<double, int32_t>(A, batch, lam, x, gv, st);
  } else {
    if (A->rowptr_type == SLA_I64) launch_grad<float, int64_t>(A, batch, lam, x, gv, st);
    else launch_grad<float, int32_t>(A, batch, lam, x, gv, st);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

}  // namespace sla

using namespace sla;

extern "C" {

const char *sla_status_string(int32_t status) {
  switch (status) {
    case SLA_OK: return "SLA_OK";
    case SLA_NOT_CONVERGED: return "SLA_NOT_CONVERGED";
    case SLA_BREAKDOWN: return "SLA_BREAKDOWN";
    case SLA_INVALID_ARG: return "SLA_INVALID_ARG";
    case SLA_BAD_CSR: return "SLA_BAD_CSR";
    case SLA_NONFINITE: return "SLA_NONFINITE";
    case SLA_WORKSPACE_TOO_SMALL: return "SLA_WORKSPACE_TOO_SMALL";
    case SLA_TIMEOUT: return "SLA_TIMEOUT";
    case SLA_CUDA_ERROR: return "SLA_CUDA_ERROR";
    default: return "SLA_UNKNOWN_STATUS";
  }
}

const char *sla_last_cuda_error(void) { return cudaGetErrorString(t_last_error); }

int32_t sla_version(void) { return 100; }

uint64_t sla_launch_count(void) { return g_launches.load(); }

size_t sla_cg_workspace_bytes(int64_t n, int64_t batch, int32_t dtype, int32_t precond) {
  if (n < 0 || batch < 1 || (dtype != SLA_F32 && dtype != SLA_F64)) return 0;
  if (precond != SLA_PRECOND_NONE && precond != SLA_PRECOND_JACOBI) return 0;
  return workspace_bytes(n, batch, dtype, precond);
}

sla_status sla_validate_csr(const sla_csr *A, int32_t check_symmetric, int64_t *bad_row, void *workspace,
                            size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, check_symmetric != 0));
  if (!workspace || ws_bytes < 256 || !aligned(workspace, 256)) return SLA_INVALID_ARG;
  if (bad_row) *bad_row = -1;
  if (A->n == 0) return A->nnz == 0 ? SLA_OK : SLA_BAD_CSR;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned long long *flag = (unsigned long long *)workspace;
  cudaError_t e = cudaMemsetAsync(flag, 0xff, sizeof(unsigned long long), st);
  if (e != cudaSuccess) return fail(e);
  const int grid = grid_for(A->n, kBlock * 4);
  if (A->rowptr_type == SLA_I64)
    validate_kernel<int64_t><<<grid, kBlock, 0, st>>>(A->n, A->nnz, (const int64_t *)A->row_ptr, A->col_idx,
                                                      A->values, A->dtype, check_symmetric, flag);
  else
    validate_kernel<int32_t><<<grid, kBlock, 0, st>>>(A->n, A->nnz, (const int32_t *)A->row_ptr, A->col_idx,
                                                      A->values, A->dtype, check_symmetric, flag);
  count_launches(1);
  unsigned long long h = 0;
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
  if ((e = cudaMemcpyAsync(&h, flag, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
  if (h == ~0ull) return SLA_OK;
  if (bad_row) *bad_row = (int64_t)h;
  return SLA_BAD_CSR;
}

sla_status sla_spmv(const sla_csr *A, const void *x, void *y, void *stream) {
  SLA_CHECK(check_csr(A, true));
  SLA_CHECK(check_vec(x, A, false));
  SLA_CHECK(check_vec(y, A, false));
  if (A->n == 0) return SLA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) launch_spmv<double, int64_t>(A, x, y, st);
    else launch_spmv<double, int32_t>(A, x, y, st);
  } else {
    if (A->rowptr_type == SLA_I64) launch_spmv<float, int64_t>(A, x, y, st);
    else launch_spmv<float, int32_t>(A, x, y, st);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

sla_status sla_grad_values(const sla_csr *A, const void *lambda, const void *x, void *grad_values, void *stream) {
  SLA_CHECK(check_csr(A, false));
  SLA_CHECK(check_vec(lambda, A, false));
  SLA_CHECK(check_vec(x, A, false));
  if (A->nnz > 0 && !grad_values) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(grad_values, A, true));
  return grad_values_entry(A, 1, lambda, x, grad_values, (cudaStream_t)stream);
}

sla_status sla_matvec_grad_values(const sla_csr *A, const void *gy, const void *x, void *grad_values,
                                  void *stream) {
  SLA_CHECK(check_csr(A, false));
  SLA_CHECK(check_vec(gy, A, false));
  SLA_CHECK(check_vec(x, A, false));
  if (A->nnz > 0 && !grad_values) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(grad_values, A, true));
  if (A->n == 0 || A->nnz == 0) return SLA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int g = pattern_grid(A->n);
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64)
      matvec_grad_kernel<double, int64_t><<<g, kPatBlock, 0, st>>>(A->n, A->nnz, (const int64_t *)A->row_ptr,
                                                                    A->col_idx, (const double *)gy,
                                                                    (const double *)x, (double *)grad_values);
    else
      matvec_grad_kernel<double, int32_t><<<g, kPatBlock, 0, st>>>(A->n, A->nnz, (const int32_t *)A->row_ptr,
                                                                    A->col_idx, (const double *)gy,
                                                                    (const double *)x, (double *)grad_values);
  } else {
    if (A->rowptr_type == SLA_I64)
      matvec_grad_kernel<float, int64_t><<<g, kPatBlock, 0, st>>>(A->n, A->nnz, (const int64_t *)A->row_ptr,
                                                                   A->col_idx, (const float *)gy, (const float *)x,
                                                                   (float *)grad_values);
    else
      matvec_grad_kernel<float, int32_t><<<g, kPatBlock, 0, st>>>(A->n, A->nnz, (const int32_t *)A->row_ptr,
                                                                   A->col_idx, (const float *)gy, (const float *)x,
                                                                   (float *)grad_values);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

sla_status sla_spmv_transpose(const sla_csr *A, const void *x, void *y, uint32_t *bad, void *stream) {
  SLA_CHECK(check_csr(A, true));
  SLA_CHECK(check_vec(x, A, false));
  SLA_CHECK(check_vec(y, A, false));
  if (!aligned(bad, 4)) return SLA_INVALID_ARG;
  if (A->n == 0) return SLA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int g = grid_for(A->n, kBlock * 4);
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64)
      spmv_t_kernel<double, int64_t><<<g, kBlock, 0, st>>>(A->n, A->nnz, (const int64_t *)A->row_ptr, A->col_idx,
                                                            (const double *)A->values, (const double *)x,
                                                            (double *)y, bad);
    else
      spmv_t_kernel<double, int32_t><<<g, kBlock, 0, st>>>(A->n, A->nnz, (const int32_t *)A->row_ptr, A->col_idx,
                                                            (const double *)A->values, (const double *)x,
                                                            (double *)y, bad);
  } else {
    if (A->rowptr_type == SLA_I64)
      spmv_t_kernel<float, int64_t><<<g, kBlock, 0, st>>>(A->n, A->nnz, (const int64_t *)A->row_ptr, A->col_idx,
                                                           (const float *)A->values, (const float *)x, (float *)y,
                                                           bad);
    else
      spmv_t_kernel<float, int32_t><<<g, kBlock, 0, st>>>(A->n, A->nnz, (const int32_t *)A->row_ptr, A->col_idx,
                                                           (const float *)A->values, (const float *)x, (float *)y,
                                                           bad);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

sla_status sla_cg_solve(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *opts, void *x,
                        sla_cg_info *info, double *history, void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, true));
  SLA_CHECK(check_opts(opts));
  SLA_CHECK(check_vec(b, A, false));
  SLA_CHECK(check_vec(x0, A, true));
  SLA_CHECK(check_vec(x, A, false));
  if (history && !aligned(history, 8)) return SLA_INVALID_ARG;
  if (A->n == 0) {
    fill_empty(info, 1);
    if (history) {
      cudaError_t e = cudaMemsetAsync(history, 0, sizeof(double), (cudaStream_t)stream);
      if (e != cudaSuccess) return fail(e);
    }
    return SLA_OK;
  }
  SLA_CHECK(check_ws(A, 1, opts, workspace, ws_bytes));
  return cg_entry(A, 1, A->values, 0, b, x0, opts, x, info, history, workspace, (cudaStream_t)stream);
}

sla_status sla_cg_adjoint(const sla_csr *A, const void *x, const void *g, const sla_cg_opts *opts, void *grad_b,
                          void *grad_values, sla_cg_info *info, void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, true));
  SLA_CHECK(check_opts(opts));
  SLA_CHECK(check_vec(x, A, false));
  SLA_CHECK(check_vec(g, A, false));
  SLA_CHECK(check_vec(grad_b, A, false));
  SLA_CHECK(check_vec(grad_values, A, true));
  if (A->n == 0) {
    fill_empty(info, 1);
    return SLA_OK;
  }
  SLA_CHECK(check_ws(A, 1, opts, workspace, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  // lambda = A^{-T} g = A^{-1} g (A symmetric), written straight into grad_b.  The gradient
  // kernel is enqueued before the status is read so the host waits only once.
  sla_status s = cg_entry(A, 1, A->values, 0, g, nullptr, opts, grad_b, nullptr, nullptr, workspace, st);
  if (s != SLA_OK) return s;
  if (grad_values) SLA_CHECK(grad_values_entry(A, 1, grad_b, x, grad_values, st));
  if (!info) return SLA_OK;
  const Layout L = make_layout(A->n, 1, A->dtype == SLA_F64 ? 8 : 4, opts->precond == SLA_PRECOND_JACOBI);
  return read_info((const Ctl *)((char *)workspace + L.ctl), (const Glob *)((char *)workspace + L.glob), 1, st,
                   info);
}

sla_status sla_cg_solve_batched(const sla_csr *pattern, int64_t batch, const void *values, const void *b,
                                const void *x0, const sla_cg_opts *opts, void *x, sla_cg_info *info,
                                double *history, void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(pattern, false));
  SLA_CHECK(check_opts(opts));
  if (batch < 0 || batch > 65535) return SLA_INVALID_ARG;
  if (batch == 0) return SLA_OK;
  if (pattern->nnz > 0 && !values) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(values, pattern, true));
  SLA_CHECK(check_vec(b, pattern, false));
  SLA_CHECK(check_vec(x0, pattern, true));
  SLA_CHECK(check_vec(x, pattern, false));
  if (history && !aligned(history, 8)) return SLA_INVALID_ARG;
  if (pattern->n == 0) {
    fill_empty(info, batch);
    return SLA_OK;
  }
  SLA_CHECK(check_ws(pattern, batch, opts, workspace, ws_bytes));
  return cg_entry(pattern, batch, values, pattern->nnz, b, x0, opts, x, info, history, workspace,
                  (cudaStream_t)stream);
}

sla_status sla_cg_adjoint_batched(const sla_csr *pattern, int64_t batch, const void *values, const void *x,
                                  const void *g, const sla_cg_opts *opts, void *grad_b, void *grad_values,
                                  sla_cg_info *info, void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(pattern, false));
  SLA_CHECK(check_opts(opts));
  if (batch < 0 || batch > 65535) return SLA_INVALID_ARG;
  if (batch == 0) return SLA_OK;
  if (pattern->nnz > 0 && !values) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(values, pattern, true));
  SLA_CHECK(check_vec(x, pattern, false));
  SLA_CHECK(check_vec(g, pattern, false));
  SLA_CHECK(check_vec(grad_b, pattern, false));
  SLA_CHECK(check_vec(grad_values, pattern, true));
  if (pattern->n == 0) {
    fill_empty(info, batch);
    return SLA_OK;
  }
  SLA_CHECK(check_ws(pattern, batch, opts, workspace, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  sla_status s = cg_entry(pattern, batch, values, pattern->nnz, g, nullptr, opts, grad_b, nullptr, nullptr,
                          workspace, st);
  if (s != SLA_OK) return s;
  if (grad_values) SLA_CHECK(grad_values_entry(pattern, batch, grad_b, x, grad_values, st));
  if (!info) return SLA_OK;
  const Layout L = make_layout(pattern->n, batch, pattern->dtype == SLA_F64 ? 8 : 4,
                               opts->precond == SLA_PRECOND_JACOBI);
  return read_info((const Ctl *)((char *)workspace + L.ctl), (const Glob *)((char *)workspace + L.glob), batch,
                   st, info);
}

}  // extern "C"
