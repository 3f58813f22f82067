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

#include <algorithm>
#include <cmath>
#include <numeric>
#include <vector>

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

// ------------------------------------------------------------------------ k smallest eigenpairs
//
// Block inverse iteration with a Rayleigh-Ritz step (subspace iteration on A^{-1}; Golub and Van
// Loan, Matrix Computations, "orthogonal iteration" and the Rayleigh-Ritz procedure).  A block
// of k vectors is stored one vector after the other ([k][n]).  Per outer step:
//   W = A X; H = X^T W; H = Q diag(theta) Q^T (theta ascending); X <- X Q, W <- W Q (Ritz pairs);
//   residuals ||W_s - theta_s X_s||; then Y = A^{-1} X by the batched CG (k right-hand sides, one
//   matrix: values stride 0) from Y = X diag(1 / theta), and X <- Y orthonormalised (Cholesky QR,
//   twice).  The n-sized work runs in the kernels below; the k x k eigenproblem and Cholesky
//   factor (k <= 16) are solved by the host, between steps, in fp64.

// Y[s] = A X[s] for the vectors s = blockIdx.y: row sums in storage order with fused multiply-adds.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) eigk_spmm(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                    const int32_t *__restrict__ ci, const V *__restrict__ val,
                                                    const V *__restrict__ X, V *__restrict__ Y, uint32_t *bad) {
  const int64_t o = (int64_t)blockIdx.y * n;
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, i, nnz, e0, e1, bad);
    V acc = V(0);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t c = ci[e];
      if (col_ok(c, (int32_t)n, bad)) acc = fmav<V>(val[e], X[o + c], acc);
    }
    Y[o + i] = acc;
  }
}

// Block partials of <X[a], Y[b]> for a = blockIdx.y and every b in [a, k): slot a * k + b.
template <typename V>
__global__ void __launch_bounds__(kBlock) eigk_dots(int64_t n, int k, const V *__restrict__ X,
                                                    const V *__restrict__ Y, double *part) {
  const int a = blockIdx.y;
  double acc[kEigMaxVecs];
#pragma unroll
  for (int b = 0; b < kEigMaxVecs; ++b) acc[b] = 0.0;
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    const double xa = (double)X[(int64_t)a * n + i];
#pragma unroll
    for (int b = 0; b < kEigMaxVecs; ++b)
      if (b >= a && b < k) acc[b] = fma(xa, (double)Y[(int64_t)b * n + i], acc[b]);
  }
#pragma unroll
  for (int b = 0; b < kEigMaxVecs; ++b) {
    if (b < a || b >= k) continue;  // uniform over the block
    double v[1] = {acc[b]};
    block_sum<1>(v);
    if (threadIdx.x == 0) part[(size_t)(a * k + b) * kMaxBlocksPerSystem + blockIdx.x] = v[0];
  }
}

// Block partials of ||W[s] - theta_s X[s]||^2 (slot 2s) and sum_i X[s][i] (slot 2s + 1), s = blockIdx.y.
template <typename V>
__global__ void __launch_bounds__(kBlock) eigk_resid(int64_t n, const V *__restrict__ X, const V *__restrict__ W,
                                                     const double *__restrict__ theta, double *part) {
  const int s = blockIdx.y;
  const double th = theta[s];
  const int64_t o = (int64_t)s * n;
  double acc[2] = {0.0, 0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    const double x = (double)X[o + i];
    const double r = fma(-th, x, (double)W[o + i]);
    acc[0] = fma(r, r, acc[0]);
    acc[1] += x;
  }
  block_sum<2>(acc);
  if (threadIdx.x == 0) {
    part[(size_t)(2 * s) * kMaxBlocksPerSystem + blockIdx.x] = acc[0];
    part[(size_t)(2 * s + 1) * kMaxBlocksPerSystem + blockIdx.x] = acc[1];
  }
}

// out[slot] = the G partials of slot blockIdx.x added in a fixed order (lane l: l, l + 32, ...,
// then a shuffle tree); slots a block did not write are left alone by the caller.
__global__ void eigk_reduce(int G, const double *__restrict__ part, double *__restrict__ out, const int *slots) {
  const int slot = slots[blockIdx.x];
  double t = 0.0;
  for (int i = threadIdx.x; i < G; i += 32) t += __ldcg(part + (size_t)slot * kMaxBlocksPerSystem + i);
  t = warp_sum(t);
  if (threadIdx.x == 0) out[blockIdx.x] = t;
}

// Z[s] = sum_t X[t] * M[t][s] (M row-major k x k, fp64; sum over t in order), s = blockIdx.y.
template <typename V>
__global__ void __launch_bounds__(kBlock) eigk_combine(int64_t n, int k, const V *__restrict__ X,
                                                       const double *__restrict__ M, V *__restrict__ Z) {
  const int s = blockIdx.y;
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    double acc = 0.0;
    for (int t = 0; t < k; ++t) acc = fma((double)X[(int64_t)t * n + i], M[t * k + s], acc);
    Z[(int64_t)s * n + i] = (V)acc;
  }
}

// Symmetric k x k eigenproblem H = Q diag(theta) Q^T by cyclic Jacobi rotations (Golub and Van
// Loan, "the cyclic Jacobi algorithm"), theta ascending, Q's columns the eigenvectors (row-major).
void sym_eig_small(int k, std::vector<double> H, std::vector<double> &theta, std::vector<double> &Q) {
  Q.assign((size_t)k * k, 0.0);
  for (int i = 0; i < k; ++i) Q[(size_t)i * k + i] = 1.0;
  auto h = [&](int r, int c) -> double & { return H[(size_t)r * k + c]; };
  for (int sweep = 0; sweep < 100; ++sweep) {
    double off = 0.0, tot = 0.0;
    for (int r = 0; r < k; ++r)
      for (int c = 0; c < k; ++c) {
        tot += h(r, c) * h(r, c);
        if (r != c) off += h(r, c) * h(r, c);
      }
    if (off <= 1e-32 * tot || off == 0.0) break;
    for (int p = 0; p < k - 1; ++p)
      for (int q = p + 1; q < k; ++q) {
        const double apq = h(p, q);
        if (apq == 0.0) continue;
        const double tau = (h(q, q) - h(p, p)) / (2.0 * apq);
        const double t = (tau >= 0.0 ? 1.0 : -1.0) / (std::fabs(tau) + std::sqrt(1.0 + tau * tau));
        const double c = 1.0 / std::sqrt(1.0 + t * t), sn = t * c;
        for (int r = 0; r < k; ++r) {  // H <- H J (columns p, q)
          const double hp = h(r, p), hq = h(r, q);
          h(r, p) = c * hp - sn * hq;
          h(r, q) = sn * hp + c * hq;
        }
        for (int r = 0; r < k; ++r) {  // H <- J^T H (rows p, q)
          const double hp = h(p, r), hq = h(q, r);
          h(p, r) = c * hp - sn * hq;
          h(q, r) = sn * hp + c * hq;
        }
        for (int r = 0; r < k; ++r) {  // Q <- Q J
          const double qp = Q[(size_t)r * k + p], qq = Q[(size_t)r * k + q];
          Q[(size_t)r * k + p] = c * qp - sn * qq;
          Q[(size_t)r * k + q] = sn * qp + c * qq;
        }
      }
  }
  std::vector<int> ord(k);
  std::iota(ord.begin(), ord.end(), 0);
  std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return h(a, a) < h(b, b); });
  std::vector<double> Qs((size_t)k * k);
  theta.assign(k, 0.0);
  for (int j = 0; j < k; ++j) {
    theta[j] = h(ord[j], ord[j]);
    for (int r = 0; r < k; ++r) Qs[(size_t)r * k + j] = Q[(size_t)r * k + ord[j]];
  }
  Q.swap(Qs);
}

// G = R^T R with R upper triangular (Cholesky); Rinv = R^{-1}.  False when G is not positive
// definite to working precision (the block lost rank).
bool chol_inv_small(int k, const std::vector<double> &G, std::vector<double> &Rinv) {
  std::vector<double> R((size_t)k * k, 0.0);
  for (int j = 0; j < k; ++j) {
    double d = G[(size_t)j * k + j];
    for (int t = 0; t < j; ++t) d -= R[(size_t)t * k + j] * R[(size_t)t * k + j];
    if (!(d > 0.0) || !std::isfinite(d)) return false;
    const double rjj = std::sqrt(d);
    R[(size_t)j * k + j] = rjj;
    for (int c = j + 1; c < k; ++c) {
      double v = G[(size_t)j * k + c];
      for (int t = 0; t < j; ++t) v -= R[(size_t)t * k + j] * R[(size_t)t * k + c];
      R[(size_t)j * k + c] = v / rjj;
    }
  }
  Rinv.assign((size_t)k * k, 0.0);
  for (int c = 0; c < k; ++c) {  // column c of R^{-1} by back substitution of R y = e_c
    for (int r = c; r >= 0; --r) {
      double v = (r == c) ? 1.0 : 0.0;
      for (int t = r + 1; t <= c; ++t) v -= R[(size_t)r * k + t] * Rinv[(size_t)t * k + c];
      Rinv[(size_t)r * k + c] = v / R[(size_t)r * k + r];
    }
  }
  return true;
}

// Workspace of sla_eigsh: the batched inner CG's (k systems), three k-vector blocks, the
// reductions' partials, and the small matrices the host hands to the kernels.
struct EigkLayout {
  size_t cg, b1, b2, b3, part, small, slots, bad, total;
};

EigkLayout eigk_layout(int64_t n, int64_t k, int dtype, int precond) {
  const size_t vsz = dtype == SLA_F64 ? 8 : 4;
  EigkLayout L;
  size_t off = 0;
  L.cg = off; off += align256(workspace_bytes(n, k, dtype, precond));
  L.b1 = off; off += align256(vsz * (size_t)n * (size_t)k);
  L.b2 = off; off += align256(vsz * (size_t)n * (size_t)k);
  L.b3 = off; off += align256(vsz * (size_t)n * (size_t)k);
  L.part = off; off += align256(sizeof(double) * (size_t)kEigMaxVecs * kEigMaxVecs * kMaxBlocksPerSystem);
  L.small = off; off += align256(sizeof(double) * (size_t)(kEigMaxVecs * kEigMaxVecs + kEigMaxVecs));
  L.slots = off; off += align256(sizeof(int) * (size_t)kEigMaxVecs * kEigMaxVecs);
  L.bad = off; off += align256(sizeof(uint32_t));
  L.total = off;
  return L;
}

template <typename V, typename I>
sla_status eigk_run(const sla_csr *A, int k, V *Vout, double *mu, const sla_eig_opts *o, sla_eig_info *info,
                    char *ws, cudaStream_t st) {
  const int64_t n = A->n;
  const EigkLayout L = eigk_layout(n, k, A->dtype, o->precond);
  V *buf[4] = {Vout, (V *)(ws + L.b1), (V *)(ws + L.b2), (V *)(ws + L.b3)};
  double *part = (double *)(ws + L.part);
  double *dM = (double *)(ws + L.small);
  double *dtheta = dM + kEigMaxVecs * kEigMaxVecs;
  int *dslots = (int *)(ws + L.slots);
  uint32_t *dbad = (uint32_t *)(ws + L.bad);  // a row range or column out of bounds was skipped
  const I *rp = (const I *)A->row_ptr;
  const V *val = (const V *)A->values;
  const int G = eig_grid(n);
  cudaError_t e = cudaMemsetAsync(dbad, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return fail(e);
  info->iters = 0;
  info->inner_iters = 0;
  info->mu = 0.0;
  info->residual = 0.0;
  info->pad = 0;
  uint64_t launches = 0;
  std::vector<double> red((size_t)k * k), M;
  std::vector<int> slots;
  // runs the fixed-order reduction of the listed slots into red[0 .. slots.size())
  auto reduce = [&](const std::vector<int> &sl) -> cudaError_t {
    cudaError_t er = cudaMemcpyAsync(dslots, sl.data(), sizeof(int) * sl.size(), cudaMemcpyHostToDevice, st);
    if (er != cudaSuccess) return er;
    eigk_reduce<<<(unsigned)sl.size(), 32, 0, st>>>(G, part, dM, dslots);
    ++launches;
    if ((er = cudaGetLastError()) != cudaSuccess) return er;
    if ((er = cudaMemcpyAsync(red.data(), dM, sizeof(double) * sl.size(), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
      return er;
    return cudaStreamSynchronize(st);
  };
  // Gram matrix X^T Y (symmetric by construction when Y = A X or Y = X) into Hm
  auto gram = [&](const V *X, const V *Y, std::vector<double> &Hm) -> cudaError_t {
    eigk_dots<V><<<dim3(G, k), kBlock, 0, st>>>(n, k, X, Y, part);
    ++launches;
    cudaError_t er = cudaGetLastError();
    if (er != cudaSuccess) return er;
    slots.clear();
    for (int a = 0; a < k; ++a)
      for (int b = a; b < k; ++b) slots.push_back(a * k + b);
    if ((er = reduce(slots)) != cudaSuccess) return er;
    Hm.assign((size_t)k * k, 0.0);
    for (size_t q = 0; q < slots.size(); ++q) {
      const int a = slots[q] / k, b = slots[q] % k;
      Hm[(size_t)a * k + b] = Hm[(size_t)b * k + a] = red[q];
    }
    return cudaSuccess;
  };
  // Z = X M (M host, k x k row-major)
  auto combine = [&](const V *X, const std::vector<double> &Mh, V *Z) -> cudaError_t {
    cudaError_t er = cudaMemcpyAsync(dM, Mh.data(), sizeof(double) * (size_t)k * k, cudaMemcpyHostToDevice, st);
    if (er != cudaSuccess) return er;
    eigk_combine<V><<<dim3(G, k), kBlock, 0, st>>>(n, k, X, dM, Z);
    ++launches;
    return cudaGetLastError();
  };
  // X <- X orthonormalised by Cholesky QR twice, through the scratch block T; false: lost rank
  auto orthonormalise = [&](V *X, V *T, bool &ok) -> cudaError_t {
    std::vector<double> Gm, Rinv;
    ok = true;
    V *src = X, *dst = T;
    for (int pass = 0; pass < 2; ++pass) {
      cudaError_t er = gram(src, src, Gm);
      if (er != cudaSuccess) return er;
      if (!chol_inv_small(k, Gm, Rinv)) {
        ok = false;
        return cudaSuccess;
      }
      if ((er = combine(src, Rinv, dst)) != cudaSuccess) return er;
      std::swap(src, dst);
    }
    return cudaSuccess;  // two passes: the result is back in X
  };
  int32_t status = SLA_NOT_CONVERGED;
  int cur = 0, wb = 1, t1 = 2, t2 = 3;  // basis, its image A X, two scratch blocks
  bool ok = true;
  if ((e = orthonormalise(buf[cur], buf[t1], ok)) != cudaSuccess) return fail(e);
  std::vector<double> H, theta, Q, resid(k), vsum(k);
  int64_t it = 0;
  if (!ok) status = SLA_BREAKDOWN;
  while (ok) {
    eigk_spmm<V, I><<<dim3(G, k), kBlock, 0, st>>>(n, A->nnz, rp, A->col_idx, val, buf[cur], buf[wb], dbad);
    ++launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    if ((e = gram(buf[cur], buf[wb], H)) != cudaSuccess) return fail(e);
    uint32_t hbad = 0;
    if ((e = cudaMemcpyAsync(&hbad, dbad, sizeof(hbad), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)
      return fail(e);
    if (hbad) { status = SLA_BAD_CSR; break; }
    bool finite = true;
    for (double v : H) finite = finite && std::isfinite(v);
    if (!finite) { status = SLA_NONFINITE; break; }
    sym_eig_small(k, H, theta, Q);
    // Ritz vectors and their images
    if ((e = combine(buf[cur], Q, buf[t1])) != cudaSuccess) return fail(e);
    if ((e = combine(buf[wb], Q, buf[t2])) != cudaSuccess) return fail(e);
    std::swap(cur, t1);
    std::swap(wb, t2);
    if ((e = cudaMemcpyAsync(dtheta, theta.data(), sizeof(double) * k, cudaMemcpyHostToDevice, st)) != cudaSuccess)
      return fail(e);
    eigk_resid<V><<<dim3(G, k), kBlock, 0, st>>>(n, buf[cur], buf[wb], dtheta, part);
    ++launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    slots.clear();
    for (int s = 0; s < 2 * k; ++s) slots.push_back(s);
    if ((e = reduce(slots)) != cudaSuccess) return fail(e);
    double rmax = 0.0, rel_max = 0.0;
    bool conv = true;
    for (int s = 0; s < k; ++s) {
      resid[s] = std::sqrt(std::max(red[2 * s], 0.0));
      vsum[s] = red[2 * s + 1];
      rmax = std::max(rmax, resid[s]);
      if (theta[s] > 0.0) rel_max = std::max(rel_max, resid[s] / theta[s]);
      conv = conv && resid[s] <= o->tol * theta[s];
    }
    info->mu = theta[0];
    info->residual = rmax;
    if (!std::isfinite(rmax)) { status = SLA_NONFINITE; break; }
    if (!(theta[0] > 0.0)) { status = SLA_BREAKDOWN; break; }
    if (conv) { status = SLA_OK; break; }
    if (it >= o->maxit) { status = SLA_NOT_CONVERGED; break; }
    // Y = A^{-1} X from Y = X diag(1/theta), every vector to the rtol inner_factor * max_s
    // residual_s / theta_s (per-vector tolerances, tighter for the vectors nearer convergence,
    // took about a quarter more CG iterations for the same outer steps).  When one system fits
    // the resident engine the k solves run one after another there; otherwise together in the
    // batched CG (one matrix: values stride 0).
    M.assign((size_t)k * k, 0.0);
    for (int s = 0; s < k; ++s) M[(size_t)s * k + s] = 1.0 / theta[s];
    if ((e = combine(buf[cur], M, buf[t1])) != cudaSuccess) return fail(e);
    sla_cg_opts co;
    co.rtol = o->inner_factor * rel_max;
    co.maxit = o->inner_maxit;
    co.precond = (sla_precond)o->precond;
    co.unroll = 0;
    co.loop = o->loop;
    co.reserved = 0;
    std::vector<sla_cg_info> ci((size_t)k);
    const bool one_by_one = (o->loop == SLA_LOOP_AUTO || o->loop == SLA_LOOP_RESIDENT) &&
                            resident_fits(n, 1, A->dtype, o->precond, o->inner_maxit);
    if (one_by_one) {
      const size_t vb = sizeof(V) * (size_t)n;
      for (int s = 0; s < k; ++s) {
        const char *xs = (const char *)buf[cur] + vb * s;
        char *ys = (char *)buf[t1] + vb * s;
        const sla_status cs = cg_entry(A, 1, A->values, 0, xs, ys, &co, ys, &ci[s], nullptr, ws + L.cg, st);
        if (cs != SLA_OK) return cs;
      }
    } else {
      const sla_status cs = cg_entry(A, k, A->values, 0, buf[cur], buf[t1], &co, buf[t1], ci.data(), nullptr,
                                     ws + L.cg, st);
      if (cs != SLA_OK) return cs;
    }
    int32_t inner_bad = SLA_OK;
    for (int s = 0; s < k; ++s) {
      info->inner_iters += ci[s].iters;
      if (ci[s].status != SLA_OK && ci[s].status != SLA_NOT_CONVERGED) inner_bad = ci[s].status;
    }
    ++it;
    if (inner_bad != SLA_OK) { status = inner_bad; break; }
    // the new basis: Y orthonormalised, into the basis block
    std::swap(cur, t1);
    if ((e = orthonormalise(buf[cur], buf[t2], ok)) != cudaSuccess) return fail(e);
    if (!ok) status = SLA_BREAKDOWN;
  }
  info->iters = it;
  info->status = status;
  // the eigenvectors into the caller's block, each with sum_i v_i >= 0
  if (status == SLA_OK || status == SLA_NOT_CONVERGED) {
    M.assign((size_t)k * k, 0.0);
    for (int s = 0; s < k; ++s) M[(size_t)s * k + s] = vsum[s] < 0.0 ? -1.0 : 1.0;
    // into the caller's block directly, or through a scratch block when the basis is already there
    const int dst = cur == 0 ? t1 : 0;
    if ((e = combine(buf[cur], M, buf[dst])) != cudaSuccess) return fail(e);
    if (dst != 0 &&
        (e = cudaMemcpyAsync(Vout, buf[dst], sizeof(V) * (size_t)n * k, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
      return fail(e);
    for (int s = 0; s < k; ++s) mu[s] = theta[s];
  } else if (cur != 0) {
    if ((e = cudaMemcpyAsync(Vout, buf[cur], sizeof(V) * (size_t)n * k, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
      return fail(e);
  }
  count_launches(launches);
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

size_t sla_eigsh_workspace_bytes(int64_t n, int64_t k, int32_t dtype, int32_t precond) {
  if (n < 0 || k < 1 || k > kEigMaxVecs || (dtype != SLA_F32 && dtype != SLA_F64)) return 0;
  if (precond != SLA_PRECOND_NONE && precond != SLA_PRECOND_JACOBI) return 0;
  return eigk_layout(n, k, dtype, precond).total;
}

sla_status sla_eigsh(const sla_csr *A, int64_t k, void *V, double *mu, const sla_eig_opts *opts, sla_eig_info *info,
                     void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, true));
  if (!eig_opts_ok(opts) || !info || !mu) return SLA_INVALID_ARG;
  if (k < 1 || k > kEigMaxVecs || k > A->n) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(V, A, false));
  if (!workspace || !aligned(workspace, 256)) return SLA_INVALID_ARG;
  if (ws_bytes < eigk_layout(A->n, k, A->dtype, opts->precond).total) return SLA_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  char *ws = (char *)workspace;
  const int kk = (int)k;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) return eigk_run<double, int64_t>(A, kk, (double *)V, mu, opts, info, ws, st);
    return eigk_run<double, int32_t>(A, kk, (double *)V, mu, opts, info, ws, st);
  }
  if (A->rowptr_type == SLA_I64) return eigk_run<float, int64_t>(A, kk, (float *)V, mu, opts, info, ws, st);
  return eigk_run<float, int32_t>(A, kk, (float *)V, mu, opts, info, ws, st);
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
