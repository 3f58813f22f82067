// Eigenvalue problems: the smallest eigenpair of a symmetric positive definite CSR matrix by
// inverse iteration on the library's CG, and the eigenvalue gradient on the sparsity pattern.
//
// Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers and Sparse
// Tensor Parallelism for PyTorch" (Chi, Wen), technical summary:
//   - Methodology 1 names the ".eigsh" API but no eigensolver.  Inverse iteration is taken here
//     because each of its steps is one solve with A, the operation the rest of the library makes
//     fast; the solves are inexact, with a CG tolerance proportional to the current eigen-residual
//     (inexact inverse iteration, Golub and Ye, BIT 40, 2000) and warm-started from v / mu.
//   - Methodology 2, eigenvalue problems: d mu / d A_ij = v_i v_j (Hellmann-Feynman), an outer
//     product evaluated on the stored entries only.
#include <cuda_runtime.h>

#include <cmath>

#include "sla_common.cuh"
#include "sla_host.h"
#include "sla_pattern.cuh"

namespace sla {
namespace {

constexpr int kEigMaxVecs = 16;

// Scalars of one inverse-iteration step, written by the last block of each reduction kernel.
struct EigScal {
  double yy;      // ||y||^2 of the unnormalised iterate
  double scale;   // 1 / ||y|| (0 if ||y|| is 0 or not finite)
  double mu;      // Rayleigh quotient v^T A v
  double vsum;    // sum_i v_i (sign convention)
  double rr;      // ||A v - mu v||^2
  uint32_t ticket;
  uint32_t bad;   // a row range or column index out of bounds was skipped
};

struct EigWeights {
  double w[kEigMaxVecs];
};

// Workspace of sla_eig_smallest: the inner CG's workspace first, then y, w = A v, the partial
// sums of the reductions and the step's scalars.
struct EigLayout {
  size_t cg, y, w, part, scal, total;
};

EigLayout eig_layout(int64_t n, int dtype, int precond) {
  const size_t vsz = dtype == SLA_F64 ? 8 : 4;
  EigLayout L;
  size_t off = 0;
  L.cg = off; off += align256(workspace_bytes(n, 1, dtype, precond));
  L.y = off; off += align256(vsz * (size_t)n);
  L.w = off; off += align256(vsz * (size_t)n);
  L.part = off; off += align256(sizeof(double) * 2 * kMaxBlocksPerSystem);
  L.scal = off; off += align256(sizeof(EigScal));
  L.total = off;
  return L;
}

// Blocks of the step kernels: about 4 rows per thread, at most 8 blocks per SM and never more
// partial-sum slots than the reduction scratch holds.
int eig_grid(int64_t n) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (n + 4 * kBlock - 1) / (4 * kBlock);
  if (g > (int64_t)sms * 8) g = (int64_t)sms * 8;
  if (g > kMaxBlocksPerSystem) g = kMaxBlocksPerSystem;
  return g < 1 ? 1 : (int)g;
}

// ------------------------------------------------------------------------ step kernels

// ||y||^2 and 1/||y||.
template <typename V>
__global__ void __launch_bounds__(kBlock) eig_norm(int64_t n, const V *__restrict__ y, double *part, EigScal *S) {
  double acc[1] = {0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    const double t = (double)y[i];
    acc[0] = fma(t, t, acc[0]);
  }
  block_sum<1>(acc);
  if (!publish_last<1>(acc, part, &S->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[1];
  reduce_partials<1>(part, (int)gridDim.x, &S->ticket, tot);
  if (threadIdx.x == 0) {
    S->yy = tot[0];
    S->scale = (tot[0] > 0.0 && isfinite(tot[0])) ? 1.0 / sqrt(tot[0]) : 0.0;
  }
}

// v = y / ||y||, w = A v (as (A y) / ||y||: the SpMV reads y, which no block writes here), and
// the sums v.w (the Rayleigh quotient, v having unit norm) and sum_i v_i.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) eig_apply(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                    const int32_t *__restrict__ ci, const V *__restrict__ val,
                                                    const V *__restrict__ y, V *__restrict__ v, V *__restrict__ w,
                                                    double *part, EigScal *S) {
  const double s = S->scale;
  double acc[2] = {0.0, 0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, i, nnz, e0, e1, &S->bad);
    V sum = V(0);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t c = ci[e];
      if (col_ok(c, (int32_t)n, &S->bad)) sum = fmav<V>(val[e], y[c], sum);
    }
    const V vi = (V)(s * (double)y[i]);
    const V wi = (V)(s * (double)sum);
    v[i] = vi;
    w[i] = wi;
    acc[0] = fma((double)vi, (double)wi, acc[0]);
    acc[1] += (double)vi;
  }
  block_sum<2>(acc);
  if (!publish_last<2>(acc, part, &S->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[2];
  reduce_partials<2>(part, (int)gridDim.x, &S->ticket, tot);
  if (threadIdx.x == 0) {
    S->mu = tot[0];
    S->vsum = tot[1];
  }
}

// ||w - mu v||^2, and y = v / mu: the start of the next inner solve A y = v.
template <typename V>
__global__ void __launch_bounds__(kBlock) eig_resid(int64_t n, const V *__restrict__ v, const V *__restrict__ w,
                                                    V *__restrict__ y, double *part, EigScal *S) {
  const double mu = S->mu;
  const double inv = (mu > 0.0 && isfinite(mu)) ? 1.0 / mu : 0.0;
  double acc[1] = {0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    const double vi = (double)v[i];
    const double r = fma(-mu, vi, (double)w[i]);
    acc[0] = fma(r, r, acc[0]);
    y[i] = (V)(vi * inv);
  }
  block_sum<1>(acc);
  if (!publish_last<1>(acc, part, &S->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[1];
  reduce_partials<1>(part, (int)gridDim.x, &S->ticket, tot);
  if (threadIdx.x == 0) S->rr = tot[0];
}

template <typename V>
__global__ void __launch_bounds__(kBlock) eig_negate(int64_t n, V *__restrict__ v) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock)
    v[i] = -v[i];
}

// ------------------------------------------------------------------------ gradient kernel

// gv[e] = sum_s (w_s * V_s[row(e)]) * V_s[col(e)], summed over s in order from the s = 0 term, in
// fp64 with separately rounded operations, then rounded once to V: one streaming pass over the
// pattern (sla_pattern.cuh) whose row factor w_0 * V_0[row] is formed once per row (none when
// w_0 = 1, which is exact), so that for k = 1 an entry costs one fp64 multiply.  The loop over
// further eigenvectors has a dynamic trip count: an unrolled loop with predicated-off iterations
// would still occupy the fp64 unit.
template <typename V, typename I>
__global__ void __launch_bounds__(kPatBlock, kPatMinBlocks) eig_grad_kernel(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                             const int32_t *__restrict__ ci, int k,
                                                             const V *__restrict__ vec, EigWeights W,
                                                             V *__restrict__ gv) {
  __shared__ PatSmem<double> sm;
  __shared__ double sw[kEigMaxVecs];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kEigMaxVecs; ++s) sw[s] = W.w[s];  // static indices: no local-memory copy
  }
  __syncthreads();
  const double w0 = sw[0];
  pattern_pass<double, I>(
      n, nnz, rp, ci, sm, [&](int64_t i) { return vec[i]; },
      [&](V raw) {
        const double a = (double)raw;
        return w0 == 1.0 ? a : __dmul_rn(w0, a);
      },
      [&](int32_t c) { return __ldg(vec + c); },
      [&](int64_t e, int64_t row, double wv0, int32_t c, V vc) {
        double acc = 0.0;
        if ((uint32_t)c < (uint32_t)n) {
          acc = __dmul_rn(wv0, (double)vc);
#pragma unroll 1
          for (int s = 1; s < k; ++s) {
            const double ws = sw[s];
            const double a = (double)vec[(int64_t)s * n + row];
            const double wa = ws == 1.0 ? a : __dmul_rn(ws, a);
            acc = __dadd_rn(acc, __dmul_rn(wa, (double)vec[(int64_t)s * n + c]));
          }
        }
        __stcs(gv + e, (V)acc);
      });
}

// ------------------------------------------------------------------------ host side

template <typename V, typename I>
sla_status eig_run(const sla_csr *A, V *v, const sla_eig_opts *o, sla_eig_info *info, char *ws, cudaStream_t st) {
  const int64_t n = A->n;
  const EigLayout L = eig_layout(n, A->dtype, o->precond);
  V *y = (V *)(ws + L.y);
  V *w = (V *)(ws + L.w);
  double *part = (double *)(ws + L.part);
  EigScal *S = (EigScal *)(ws + L.scal);
  const I *rp = (const I *)A->row_ptr;
  const V *val = (const V *)A->values;
  const int G = eig_grid(n);
  cudaError_t e = cudaMemsetAsync(S, 0, sizeof(EigScal), st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(y, v, sizeof(V) * (size_t)n, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return fail(e);
  info->iters = 0;
  info->inner_iters = 0;
  info->mu = 0.0;
  info->residual = 0.0;
  info->pad = 0;
  int32_t status = SLA_NOT_CONVERGED;
  EigScal h = {};
  int64_t k = 0;
  for (;;) {
    // normalise, Rayleigh quotient and residual of the current iterate
    eig_norm<V><<<G, kBlock, 0, st>>>(n, y, part, S);
    eig_apply<V, I><<<G, kBlock, 0, st>>>(n, A->nnz, rp, A->col_idx, val, y, v, w, part, S);
    eig_resid<V><<<G, kBlock, 0, st>>>(n, v, w, y, part, S);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    count_launches(3);
    if ((e = cudaMemcpyAsync(&h, S, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
    if (h.bad) { status = SLA_BAD_CSR; break; }
    if (!std::isfinite(h.yy)) { status = SLA_NONFINITE; break; }
    if (!(h.yy > 0.0)) { status = SLA_BREAKDOWN; break; }
    const double res = std::sqrt(h.rr);
    info->mu = h.mu;
    info->residual = res;
    if (!std::isfinite(h.mu) || !std::isfinite(res)) { status = SLA_NONFINITE; break; }
    if (!(h.mu > 0.0)) { status = SLA_BREAKDOWN; break; }
    if (res <= o->tol * h.mu) { status = SLA_OK; break; }
    if (k >= o->maxit) { status = SLA_NOT_CONVERGED; break; }
    // y = A^{-1} v, from y = v / mu, to a tolerance that follows the eigen-residual
    sla_cg_opts co;
    co.rtol = o->inner_factor * res / h.mu;
    co.maxit = o->inner_maxit;
    co.precond = (sla_precond)o->precond;
    co.unroll = 0;
    co.loop = o->loop;
    co.reserved = 0;
    sla_cg_info ci;
    const sla_status s = cg_entry(A, 1, A->values, 0, v, y, &co, y, &ci, nullptr, ws + L.cg, st);
    if (s != SLA_OK) return s;
    info->inner_iters += ci.iters;
    ++k;
    if (ci.status != SLA_OK && ci.status != SLA_NOT_CONVERGED) { status = ci.status; break; }
  }
  info->iters = k;
  info->status = status;
  if (h.yy > 0.0 && h.vsum < 0.0) {
    eig_negate<V><<<G, kBlock, 0, st>>>(n, v);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    count_launches(1);
  }
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
  return SLA_OK;
}

template <typename V, typename I>
sla_status eig_grad_launch(const sla_csr *A, int k, const void *vec, const EigWeights &W, void *gv,
                           cudaStream_t st) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (A->n + kPatRows - 1) / kPatRows;  // one block per row tile, at most one wave of blocks
  if (g > (int64_t)sms * kPatMinBlocks) g = (int64_t)sms * kPatMinBlocks;
  if (g < 1) g = 1;
  eig_grad_kernel<V, I><<<(unsigned)g, kPatBlock, 0, st>>>(A->n, A->nnz, (const I *)A->row_ptr, A->col_idx, k,
                                                        (const V *)vec, W, (V *)gv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

bool eig_opts_ok(const sla_eig_opts *o) {
  if (!o) return false;
  if (!(o->tol >= 0.0) || !std::isfinite(o->tol)) return false;
  if (o->maxit < 0 || o->maxit > ((int64_t)1 << 40)) return false;
  if (!(o->inner_factor > 0.0 && o->inner_factor < 1.0)) return false;
  if (o->inner_maxit < 0 || o->inner_maxit > ((int64_t)1 << 40)) return false;
  if (o->precond != SLA_PRECOND_NONE && o->precond != SLA_PRECOND_JACOBI) return false;
  if (o->loop < SLA_LOOP_AUTO || o->loop > SLA_LOOP_CLUSTER) return false;
  return true;
}

}  // namespace
}  // namespace sla

using namespace sla;

extern "C" {

size_t sla_eig_workspace_bytes(int64_t n, int32_t dtype, int32_t precond) {
  if (n < 0 || (dtype != SLA_F32 && dtype != SLA_F64)) return 0;
  if (precond != SLA_PRECOND_NONE && precond != SLA_PRECOND_JACOBI) return 0;
  return eig_layout(n, dtype, precond).total;
}

sla_status sla_eig_smallest(const sla_csr *A, void *v, const sla_eig_opts *opts, sla_eig_info *info,
                            void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, true));
  if (!eig_opts_ok(opts) || !info) return SLA_INVALID_ARG;
  if (A->n == 0) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(v, A, false));
  if (!workspace || !aligned(workspace, 256)) return SLA_INVALID_ARG;
  if (ws_bytes < eig_layout(A->n, A->dtype, opts->precond).total) return SLA_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) return eig_run<double, int64_t>(A, (double *)v, opts, info, ws, st);
    return eig_run<double, int32_t>(A, (double *)v, opts, info, ws, st);
  }
  if (A->rowptr_type == SLA_I64) return eig_run<float, int64_t>(A, (float *)v, opts, info, ws, st);
  return eig_run<float, int32_t>(A, (float *)v, opts, info, ws, st);
}

sla_status sla_eig_grad_values(const sla_csr *A, int64_t k, const void *V, const double *w, void *grad_values,
                               void *stream) {
  SLA_CHECK(check_csr(A, false));
  if (k < 0 || k > kEigMaxVecs) return SLA_INVALID_ARG;
  if (k > 0) SLA_CHECK(check_vec(V, A, false));
  if (A->nnz > 0 && !grad_values) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(grad_values, A, true));
  if (A->nnz == 0) return SLA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t vsz = A->dtype == SLA_F64 ? 8 : 4;
  if (k == 0 || A->n == 0) {
    cudaError_t e = cudaMemsetAsync(grad_values, 0, vsz * (size_t)A->nnz, st);
    return e == cudaSuccess ? SLA_OK : fail(e);
  }
  EigWeights W;
  for (int s = 0; s < kEigMaxVecs; ++s) W.w[s] = s < k ? (w ? w[s] : 1.0) : 0.0;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) return eig_grad_launch<double, int64_t>(A, (int)k, V, W, grad_values, st);
    return eig_grad_launch<double, int32_t>(A, (int)k, V, W, grad_values, st);
  }
  if (A->rowptr_type == SLA_I64) return eig_grad_launch<float, int64_t>(A, (int)k, V, W, grad_values, st);
  return eig_grad_launch<float, int32_t>(A, (int)k, V, W, grad_values, st);
}

}  // extern "C"
