/*
 * Plain fp64 CPU oracle for the differentiable CSR conjugate-gradient solve.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header or constant with the CUDA library.  It is written
 * to be read against the method's description, not to be fast: sequential
 * sums in index order, no blocking, no fusion.  Build with -ffp-contract=off so
 * that a*b+c is always a rounded multiply then a rounded add on every host
 * (x86_64 and aarch64 give identical results).
 *
 * Two builds of this one file:
 *   - plain (no OpenMP): one thread; a dot product is one sum in index order;
 *   - multi-core (-fopenmp): every loop over rows or vector entries is split
 *     across threads (each entry's arithmetic is unchanged), and a dot product
 *     is summed in fixed chunks of ORC_CHUNK entries, each chunk in index order,
 *     then the chunk sums in chunk order.  The chunk boundaries do not depend on
 *     the thread count, so this build gives the same bits on 1, 2 or N threads;
 *     it differs from the plain build only by the dot products' summation order.
 *
 * Source of the method: "torch-sla: Differentiable Sparse Linear Algebra with
 * Adjoint Solvers and Sparse Tensor Parallelism for PyTorch" (Chi, Wen),
 * technical summary:
 *   - Methodology, 1 "Unified backend abstraction": the PyTorch-native
 *     iterative solver (conjugate gradient on the GPU) and the .matvec/.solve API;
 *   - Methodology, 2 "Adjoint differentiation framework", linear systems: for
 *     Ax=b the backward solves A^T lambda = dL/dx once, and the gradient with
 *     respect to the matrix is -lambda_i x_j on the sparsity pattern only;
 *     graph O(1), memory O(n + nnz);
 *   - Methodology, 2, eigenvalue problems: d mu / d A_ij = v_i v_j
 *     (Hellmann-Feynman), an outer product on the sparsity pattern only;
 *   - Significance: the native backend uses Jacobi preconditioning.
 * The pages do not spell out the CG variant, the stopping rule or the
 * treatment of breakdown.  Readings taken here (textbook Hestenes-Stiefel CG,
 * stop when ||r_k||_2 <= rtol ||b||_2 on the recursively updated residual,
 * Jacobi M = diag(A) applied as r_i / A_ii, breakdown when p.Ap <= 0):
 *   iteration count = number of products A p inside the loop;
 *   b == 0 gives x = 0 after 0 iterations;
 *   a non-finite ||b||, r.r or p.Ap stops with status NONFINITE;
 *   p.Ap <= 0 (finite) stops with BREAKDOWN, x left at the last iterate;
 *   with Jacobi, any non-finite diagonal entry stops with NONFINITE, else any
 *   diagonal entry <= 0 or missing stops with BREAKDOWN, before the first
 *   iteration (a symmetric positive definite matrix has a positive diagonal).
 *
 * Status codes returned: 0 converged, 1 not converged after maxit, 2 breakdown,
 * 5 non-finite.
 *
 * Layout: CSR with int64 row_ptr[n+1], int32 col_idx[nnz], double values[nnz].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#define ORC_PARALLEL_FOR _Pragma("omp parallel for schedule(static)")
#else
#define ORC_PARALLEL_FOR
#endif

/* entries per dot-product chunk in the multi-core build */
#define ORC_CHUNK 4096

#define ORC_OK 0
#define ORC_NOT_CONVERGED 1
#define ORC_BREAKDOWN 2
#define ORC_NONFINITE 5

/* Threads used by the multi-core build (nthreads > 0 sets it); 1 for the plain build. */
int orc_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* y = A x: for every row, the sum over its stored entries in storage order. */
void orc_spmv(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
              const double *x, double *y) {
  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i) {
    double s = 0.0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += values[k] * x[col_idx[k]];
    y[i] = s;
  }
}

/* y = A^T x: y_j = sum over stored entries (i, j) of a_ij x_i, the entries taken row by row in
 * storage order (so each y_j adds its terms in increasing i).  n rows and n columns. */
void orc_spmv_transpose(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                        const double *x, double *y) {
  for (int64_t j = 0; j < n; ++j) y[j] = 0.0;
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) y[col_idx[k]] = y[col_idx[k]] + values[k] * x[i];
}

/* Gradient of L(y) with y = A x with respect to the stored values, for gy = dL/dy:
 * grad_values[k] = gy[row(k)] * x[col(k)] for every stored entry, in CSR order. */
void orc_matvec_grad_values(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *gy,
                            const double *x, double *grad_values) {
  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) grad_values[k] = gy[i] * x[col_idx[k]];
}

#ifndef _OPENMP
/* a . b, summed in index order. */
double orc_dot(int64_t n, const double *a, const double *b) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}
#else
/* a . b: chunk c holds entries [c*ORC_CHUNK, (c+1)*ORC_CHUNK), summed in index order; the chunk
 * sums are then added in chunk order. */
double orc_dot(int64_t n, const double *a, const double *b) {
  const int64_t nc = (n + ORC_CHUNK - 1) / ORC_CHUNK;
  double *cs = (double *)malloc(sizeof(double) * (size_t)(nc > 0 ? nc : 1));
  ORC_PARALLEL_FOR
  for (int64_t c = 0; c < nc; ++c) {
    const int64_t i1 = (c + 1) * ORC_CHUNK < n ? (c + 1) * ORC_CHUNK : n;
    double s = 0.0;
    for (int64_t i = c * ORC_CHUNK; i < i1; ++i) s += a[i] * b[i];
    cs[c] = s;
  }
  double s = 0.0;
  for (int64_t c = 0; c < nc; ++c) s += cs[c];
  free(cs);
  return s;
}
#endif

/* diag[i] = A_ii (0 when row i stores no diagonal entry). */
void orc_diagonal(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                  double *diag) {
  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i) {
    diag[i] = 0.0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k)
      if (col_idx[k] == i) diag[i] = values[k];
  }
}

/*
 * Conjugate gradient (Hestenes-Stiefel) for A x = b, optionally Jacobi
 * preconditioned (precond = 1: M = diag(A), z = M^{-1} r computed as r_i / A_ii).
 *
 *   r = b - A x0 (r = b when x0 is NULL), z = M^{-1} r, p = z, rho = r.z
 *   repeat: q = A p; alpha = rho / (p.q); x += alpha p; r -= alpha q;
 *           stop when ||r|| <= rtol ||b||; z = M^{-1} r; rho' = r.z;
 *           beta = rho'/rho; p = z + beta p; rho = rho'.
 *
 * x       : output, n entries (the last iterate on every exit).
 * history : NULL or maxit+1 entries; history[k] = ||r_k|| / ||b|| for k = 0..iters.
 * Returns the status; *iters and *rel_res (= ||r|| / ||b|| at exit) are set.
 */
int orc_cg(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
           const double *b, const double *x0, double rtol, int64_t maxit, int precond,
           double *x, double *history, int64_t *iters, double *rel_res) {
  double *r = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double *z = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double *p = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double *q = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double *d = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  int status = ORC_NOT_CONVERGED;
  *iters = 0;
  *rel_res = 0.0;

  double nb = sqrt(orc_dot(n, b, b));
  if (x0) memcpy(x, x0, sizeof(double) * (size_t)n);
  else memset(x, 0, sizeof(double) * (size_t)n);
  if (!isfinite(nb)) { status = ORC_NONFINITE; goto done; }
  if (nb == 0.0) {
    for (int64_t i = 0; i < n; ++i) x[i] = 0.0;
    if (history) history[0] = 0.0;
    status = ORC_OK;
    goto done;
  }
  if (precond == 1) {
    orc_diagonal(n, row_ptr, col_idx, values, d);
    for (int64_t i = 0; i < n; ++i)
      if (!isfinite(d[i])) { status = ORC_NONFINITE; goto done; }
    for (int64_t i = 0; i < n; ++i)
      if (!(d[i] > 0.0)) { status = ORC_BREAKDOWN; goto done; }
  }

  if (x0) {
    orc_spmv(n, row_ptr, col_idx, values, x, q);
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) r[i] = b[i] - q[i];
  } else {
    memcpy(r, b, sizeof(double) * (size_t)n);
  }
  double rr = orc_dot(n, r, r);
  *rel_res = sqrt(rr) / nb;
  if (history) history[0] = *rel_res;
  if (!isfinite(rr)) { status = ORC_NONFINITE; goto done; }
  if (sqrt(rr) <= rtol * nb) { status = ORC_OK; goto done; }

  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i) z[i] = (precond == 1) ? r[i] / d[i] : r[i];
  memcpy(p, z, sizeof(double) * (size_t)n);
  double rho = orc_dot(n, r, z);

  for (int64_t k = 0; k < maxit; ++k) {
    orc_spmv(n, row_ptr, col_idx, values, p, q);
    double pq = orc_dot(n, p, q);
    if (!isfinite(pq)) { status = ORC_NONFINITE; goto done; }
    if (!(pq > 0.0)) { status = ORC_BREAKDOWN; goto done; }
    double alpha = rho / pq;
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) x[i] = x[i] + alpha * p[i];
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) r[i] = r[i] - alpha * q[i];
    rr = orc_dot(n, r, r);
    *iters = k + 1;
    *rel_res = sqrt(rr) / nb;
    if (history) history[k + 1] = *rel_res;
    if (!isfinite(rr)) { status = ORC_NONFINITE; goto done; }
    if (sqrt(rr) <= rtol * nb) { status = ORC_OK; goto done; }
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) z[i] = (precond == 1) ? r[i] / d[i] : r[i];
    double rho_new = orc_dot(n, r, z);
    double beta = rho_new / rho;
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) p[i] = z[i] + beta * p[i];
    rho = rho_new;
  }
  status = ORC_NOT_CONVERGED;

done:
  free(r); free(z); free(p); free(q); free(d);
  return status;
}

/* grad_values[k] = -lambda[row(k)] * x[col(k)] for every stored entry, in CSR order. */
void orc_grad_values(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *lambda,
                     const double *x, double *grad_values) {
  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) grad_values[k] = -(lambda[i] * x[col_idx[k]]);
}

/*
 * Adjoint backward of x = A^{-1} b for an upstream gradient g = dL/dx:
 * lambda solves A^T lambda = g (A is symmetric here, so the same CG routine
 * with the same preconditioner, rtol and maxit, starting from lambda = 0);
 * grad_b = lambda; grad_values = -lambda_i x_j on A's pattern.
 * Returns the adjoint solve's status.
 */
int orc_cg_adjoint(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                   const double *x, const double *g, double rtol, int64_t maxit, int precond,
                   double *grad_b, double *grad_values, int64_t *iters, double *rel_res) {
  int st = orc_cg(n, row_ptr, col_idx, values, g, NULL, rtol, maxit, precond, grad_b, NULL, iters, rel_res);
  orc_grad_values(n, row_ptr, col_idx, grad_b, x, grad_values);
  return st;
}

/*
 * Eigenvalue gradient (Methodology, 2 "Adjoint differentiation framework",
 * eigenvalue problems): for a symmetric A and a unit eigenvector v of a simple
 * eigenvalue mu, the Hellmann-Feynman theorem gives d mu / d A_ij = v_i v_j, so
 * the gradient lives on the stored entries only.  For a weighted sum
 * L = sum_s w_s mu_s of k eigenvalues (eigenvectors V[s*n .. s*n+n-1]):
 *   grad_values[e] = sum over s = 0..k-1 of w_s * (v_s[i] * v_s[j])
 * for the stored entry e = (i, j): the products v_i v_j of the theorem, weighted and
 * added from zero in index order.  w == NULL means every w_s = 1.
 */
void orc_eig_grad_values(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, int64_t k, const double *V,
                         const double *w, double *grad_values) {
  ORC_PARALLEL_FOR
  for (int64_t i = 0; i < n; ++i)
    for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
      const int64_t j = col_idx[e];
      double acc = 0.0;
      for (int64_t s = 0; s < k; ++s) {
        const double ws = w ? w[s] : 1.0;
        acc = acc + ws * (V[s * n + i] * V[s * n + j]);
      }
      grad_values[e] = acc;
    }
}

/*
 * A^T as a CSR matrix (general pattern): for every column c of A, its entries taken row by row in
 * increasing row order.  tr_row_ptr: n+1; tr_col_idx, tr_values: nnz.
 */
void orc_transpose(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                   int64_t *tr_row_ptr, int32_t *tr_col_idx, double *tr_values) {
  for (int64_t c = 0; c <= n; ++c) tr_row_ptr[c] = 0;
  for (int64_t e = 0; e < row_ptr[n]; ++e) tr_row_ptr[col_idx[e] + 1] += 1;
  for (int64_t c = 0; c < n; ++c) tr_row_ptr[c + 1] += tr_row_ptr[c];
  int64_t *fill = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  for (int64_t c = 0; c < n; ++c) fill[c] = tr_row_ptr[c];
  for (int64_t i = 0; i < n; ++i)
    for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
      const int64_t c = col_idx[e];
      tr_col_idx[fill[c]] = (int32_t)i;
      tr_values[fill[c]] = values[e];
      fill[c] += 1;
    }
  free(fill);
}

/*
 * BiCGStab for a general (non-symmetric) A x = b, unpreconditioned (H. A. van der Vorst,
 * "Bi-CGSTAB", SIAM J. Sci. Stat. Comput. 13, 1992).  The torch-sla pages list BiCGStab among
 * the solvers of the .solve API; they give no variant, so the textbook one:
 *   r = b - A x0 (r = b when x0 is NULL); rhat = r (fixed shadow residual); rho_prev = alpha =
 *   omega = 1; stop at once when ||r|| <= rtol ||b||.
 *   repeat: rho = rhat.r; (rho == 0: BREAKDOWN)
 *           p = r on the first iteration, else beta = (rho / rho_prev) (alpha / omega),
 *             p = r + beta (p - omega v);
 *           v = A p; (rhat.v == 0: BREAKDOWN) alpha = rho / (rhat.v); s = r - alpha v;
 *           when ||s|| <= rtol ||b||: x = x + alpha p, r = s, stop (converged);
 *           t = A s; (t.t == 0: BREAKDOWN) omega = (t.s) / (t.t);
 *           x = (x + alpha p) + omega s; r = s - omega t;
 *           stop when ||r|| <= rtol ||b||; (omega == 0: BREAKDOWN); rho_prev = rho.
 * One iteration = one pass of the loop (two products with A).  history[k] = ||r_k|| / ||b||.
 * b == 0 gives x = 0 after 0 iterations; non-finite sums stop with NONFINITE.
 */
int orc_bicgstab(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                 const double *b, const double *x0, double rtol, int64_t maxit, double *x, double *history,
                 int64_t *iters, double *rel_res) {
  const size_t sz = sizeof(double) * (size_t)(n > 0 ? n : 1);
  double *r = (double *)malloc(sz), *rh = (double *)malloc(sz), *p = (double *)malloc(sz);
  double *v = (double *)malloc(sz), *s = (double *)malloc(sz), *t = (double *)malloc(sz);
  int status = ORC_NOT_CONVERGED;
  *iters = 0;
  *rel_res = 0.0;
  double nb = sqrt(orc_dot(n, b, b));
  if (x0) memcpy(x, x0, sizeof(double) * (size_t)n);
  else memset(x, 0, sizeof(double) * (size_t)n);
  if (!isfinite(nb)) { status = ORC_NONFINITE; goto done; }
  if (nb == 0.0) {
    for (int64_t i = 0; i < n; ++i) x[i] = 0.0;
    if (history != NULL) history[0] = 0.0;
    status = ORC_OK;
    goto done;
  }
  if (x0) {
    orc_spmv(n, row_ptr, col_idx, values, x, t);
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) r[i] = b[i] - t[i];
  } else {
    memcpy(r, b, sizeof(double) * (size_t)n);
  }
  memcpy(rh, r, sizeof(double) * (size_t)n);
  double rr = orc_dot(n, r, r);
  *rel_res = sqrt(rr) / nb;
  if (history != NULL) history[0] = *rel_res;
  if (!isfinite(rr)) { status = ORC_NONFINITE; goto done; }
  if (sqrt(rr) <= rtol * nb) { status = ORC_OK; goto done; }
  double rho_prev = 1.0, alpha = 1.0, omega = 1.0;
  for (int64_t k = 0; k < maxit; ++k) {
    const double rho = orc_dot(n, rh, r);
    if (!isfinite(rho)) { status = ORC_NONFINITE; goto done; }
    if (rho == 0.0) { status = ORC_BREAKDOWN; goto done; }
    if (k == 0) {
      memcpy(p, r, sizeof(double) * (size_t)n);
    } else {
      const double beta = (rho / rho_prev) * (alpha / omega);
      ORC_PARALLEL_FOR
      for (int64_t i = 0; i < n; ++i) p[i] = r[i] + beta * (p[i] - omega * v[i]);
    }
    orc_spmv(n, row_ptr, col_idx, values, p, v);
    const double rv = orc_dot(n, rh, v);
    if (!isfinite(rv)) { status = ORC_NONFINITE; goto done; }
    if (rv == 0.0) { status = ORC_BREAKDOWN; goto done; }
    alpha = rho / rv;
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) s[i] = r[i] - alpha * v[i];
    const double ss = orc_dot(n, s, s);
    if (!isfinite(ss)) { status = ORC_NONFINITE; goto done; }
    if (sqrt(ss) <= rtol * nb) {
      ORC_PARALLEL_FOR
      for (int64_t i = 0; i < n; ++i) x[i] += alpha * p[i];
      memcpy(r, s, sizeof(double) * (size_t)n);
      *iters = k + 1;
      *rel_res = sqrt(ss) / nb;
      if (history != NULL) history[k + 1] = *rel_res;
      status = ORC_OK;
      goto done;
    }
    orc_spmv(n, row_ptr, col_idx, values, s, t);
    const double tt = orc_dot(n, t, t);
    const double ts = orc_dot(n, t, s);
    if (!isfinite(tt) || !isfinite(ts)) { status = ORC_NONFINITE; goto done; }
    if (tt == 0.0) { status = ORC_BREAKDOWN; goto done; }
    omega = ts / tt;
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) x[i] = (x[i] + alpha * p[i]) + omega * s[i];
    ORC_PARALLEL_FOR
    for (int64_t i = 0; i < n; ++i) r[i] = s[i] - omega * t[i];
    rr = orc_dot(n, r, r);
    *iters = k + 1;
    *rel_res = sqrt(rr) / nb;
    if (history != NULL) history[k + 1] = *rel_res;
    if (!isfinite(rr)) { status = ORC_NONFINITE; goto done; }
    if (sqrt(rr) <= rtol * nb) { status = ORC_OK; goto done; }
    if (omega == 0.0) { status = ORC_BREAKDOWN; goto done; }
    rho_prev = rho;
  }
  status = ORC_NOT_CONVERGED;
done:
  free(r); free(rh); free(p); free(v); free(s); free(t);
  return status;
}

/*
 * Adjoint backward of x = A^{-1} b for a general A (Methodology, 2: A^T lambda = dL/dx, then
 * grad_b = lambda and grad_values = -lambda_i x_j on A's pattern): lambda by the same BiCGStab,
 * rtol and maxit on the explicit transpose A^T, from lambda = 0.  Returns that solve's status.
 */
int orc_bicgstab_adjoint(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const double *values,
                         const double *x, const double *g, double rtol, int64_t maxit, double *grad_b,
                         double *grad_values, int64_t *iters, double *rel_res) {
  const int64_t nnz = row_ptr[n];
  int64_t *trp = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int32_t *tci = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nnz > 0 ? nnz : 1));
  double *tv = (double *)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
  orc_transpose(n, row_ptr, col_idx, values, trp, tci, tv);
  int st = orc_bicgstab(n, trp, tci, tv, g, NULL, rtol, maxit, grad_b, NULL, iters, rel_res);
  orc_grad_values(n, row_ptr, col_idx, grad_b, x, grad_values);
  free(trp); free(tci); free(tv);
  return st;
}
