/*
 * libsla — differentiable CSR conjugate-gradient solve for one GB300 (sm_103a).
 *
 * The method is the one described in "torch-sla: Differentiable Sparse Linear
 * Algebra with Adjoint Solvers and Sparse Tensor Parallelism for PyTorch"
 * (Chi, Wen), technical summary ("TS" below):
 *   - TS Methodology 1, "Unified backend abstraction": an autograd-aware
 *     .matvec / .solve API whose GPU iterative backend is conjugate gradient;
 *     four sparse tensor kinds, among them one matrix and a batch of matrices
 *     sharing one sparsity pattern;
 *   - TS Methodology 2, "Adjoint differentiation framework", linear systems:
 *     for A x = b the backward pass solves A^T lambda = dL/dx once; the
 *     gradient with respect to the matrix is -lambda_i x_j on the sparsity
 *     pattern only, so the autograd graph is O(1) and its memory O(n + nnz),
 *     independent of the iteration count;
 *   - TS Methodology 2, eigenvalue problems: the eigenvalue gradient is the
 *     outer product v_i v_j on the sparsity pattern (Hellmann-Feynman);
 *   - TS Significance: the native iterative backend is Jacobi preconditioned.
 * Where the summary leaves a step open the library takes the textbook reading:
 * Hestenes-Stiefel CG, stopping when ||r_k||_2 <= rtol * ||b||_2 on the
 * recursively updated residual (unpreconditioned norm also under Jacobi),
 * iteration count = number of products A p in the loop, b = 0 giving x = 0.
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device (or managed) memory on the
 *     current device; "host" pointers are ordinary host memory.  The library
 *     allocates no device memory: scratch space is the caller's workspace,
 *     sized by sla_cg_workspace_bytes().  The caller keeps ownership of
 *     every buffer.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it in order.
 *   - Matrices are square CSR, canonical: row_ptr[0] = 0, row_ptr[n] = nnz,
 *     non-decreasing; within a row, col_idx strictly increasing and in
 *     [0, n); every diagonal entry stored.  The solvers assume A symmetric
 *     positive definite (so A^T = A).  sla_validate_csr() checks the
 *     structural part.
 *   - Row pointers are int32 or int64 (sla_itype); column indices int32 (so
 *     n < 2^31); values and vectors are float32 or float64 (sla_dtype), all
 *     of one type within a call.  Float32 data is updated in float32; dot
 *     products are summed in float32 over a few rows per thread and in
 *     float64 from there on, and every scalar of the iteration (alpha, beta,
 *     norms) is float64.
 *   - Kernels never read outside the caller's buffers: an out-of-range row
 *     pointer or column index is skipped (SpMV and grad_values then treat the
 *     entry as absent; a solve reports SLA_BAD_CSR).
 *   - Errors never leave a kernel waiting: invalid arguments are rejected on
 *     the host before any launch (SLA_INVALID_ARG / SLA_WORKSPACE_TOO_SMALL);
 *     numerical failures are reported through sla_cg_info.status; a CUDA
 *     runtime failure returns SLA_CUDA_ERROR (sla_last_cuda_error() names it).
 */
#ifndef SLA_H_
#define SLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SLA_API __attribute__((visibility("default")))
#else
#define SLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sla_status {
  SLA_OK = 0,                  /* converged (or nothing to do) */
  SLA_NOT_CONVERGED = 1,       /* maxit iterations done without reaching rtol; x holds the last iterate */
  SLA_BREAKDOWN = 2,           /* p.Ap <= 0, or a Jacobi diagonal <= 0: A is not SPD; x = last iterate */
  SLA_INVALID_ARG = 3,         /* null pointer, negative size, unknown enum, misaligned buffer */
  SLA_BAD_CSR = 4,             /* non-canonical CSR (sla_validate_csr), or a solve met an out-of-range
                                  row pointer or column index (such entries are skipped, never read) */
  SLA_NONFINITE = 5,           /* ||b||, r.r, p.Ap or a Jacobi diagonal is NaN or infinite */
  SLA_WORKSPACE_TOO_SMALL = 6, /* ws_bytes < sla_cg_workspace_bytes(...) */
  SLA_TIMEOUT = 7,             /* a bounded wait of the resident kernel's grid barrier expired */
  SLA_CUDA_ERROR = 8           /* a CUDA runtime call failed */
} sla_status;

typedef enum sla_dtype { SLA_F32 = 0, SLA_F64 = 1 } sla_dtype;
typedef enum sla_itype { SLA_I32 = 0, SLA_I64 = 1 } sla_itype;
typedef enum sla_precond { SLA_PRECOND_NONE = 0, SLA_PRECOND_JACOBI = 1 } sla_precond;

/* A square CSR matrix on the device (TS Methodology 1: "SparseTensor"). */
typedef struct sla_csr {
  int64_t n;              /* rows = columns, 0 <= n < 2^31 */
  int64_t nnz;            /* stored entries */
  int32_t rowptr_type;    /* sla_itype of row_ptr */
  int32_t dtype;          /* sla_dtype of values */
  const void *row_ptr;    /* device, n+1 entries */
  const int32_t *col_idx; /* device, nnz entries */
  const void *values;     /* device, nnz entries (ignored by the batched calls: values come separately) */
} sla_csr;

typedef enum sla_loop {
  SLA_LOOP_AUTO = 0,      /* CLUSTER when each system fits one thread-block cluster, else RESIDENT
                             when one system fits on chip, else GRAPH; an engine that cannot be
                             placed (its blocks not all resident at once) passes to the next */
  SLA_LOOP_HOST = 1,      /* the host launches the streaming kernels directly and reads the device
                             status every `unroll` iterations (for profilers that cannot see inside
                             conditional graphs, and for drivers without conditional nodes) */
  SLA_LOOP_GRAPH = 2,     /* streaming kernels in one CUDA graph per solve; the loop is a device-side
                             conditional WHILE node */
  SLA_LOOP_RESIDENT = 3,  /* one persistent cooperative kernel per solve, each SM keeping r and p
                             [and 1/diag] of its rows in shared memory, x and q in L2 (one system
                             whose 1/#SM share fits one SM's shared memory: about 2.0M fp64
                             unknowns on GB300, 1.3M with Jacobi); SLA_INVALID_ARG when it does not
                             fit or its blocks cannot all be resident at once */
  SLA_LOOP_CLUSTER = 4    /* one thread-block cluster (up to 16 CTAs) per system, all vectors in
                             shared memory, partner rows read through distributed shared memory,
                             hardware cluster barriers; any batch whose systems are small enough
                             (about 50K fp64 / 100K fp32 unknowns); SLA_INVALID_ARG otherwise */
} sla_loop;

typedef struct sla_cg_opts {
  double rtol;            /* stop when ||r|| <= rtol * ||b||; 0 runs exactly maxit iterations */
  int64_t maxit;          /* iteration cap, >= 0 */
  int32_t precond;        /* sla_precond */
  int32_t unroll;         /* iterations per loop body (graph) or per status read (host); 0 = default */
  int32_t loop;           /* sla_loop */
  int32_t reserved;       /* must be 0 */
} sla_cg_opts;

/* Result of one solve (host memory).  Filled after the call has synchronised the stream. */
typedef struct sla_cg_info {
  int64_t iters;          /* completed iterations (products A p inside the loop) */
  double rel_res;         /* ||r|| / ||b|| of the recursive residual at exit (0 when b = 0) */
  int32_t status;         /* sla_status of this system */
  int32_t path;           /* the sla_loop that ran: HOST, GRAPH, RESIDENT or CLUSTER */
  int64_t kernels;        /* kernel executions of this call on the GPU, counted on the device */
} sla_cg_info;

/* ---------------------------------------------------------------- housekeeping */

/* Human-readable name of a status code (static storage). */
SLA_API const char *sla_status_string(int32_t status);

/* Name of the last CUDA runtime error seen by this thread ("no error" if none). */
SLA_API const char *sla_last_cuda_error(void);

/* Library ABI version: 100 * major + minor. */
SLA_API int32_t sla_version(void);

/* Total kernels launched by this process through the library (host-side count of launches,
 * plus the device-counted kernel executions of every solve whose info was read back). */
SLA_API uint64_t sla_launch_count(void);

/*
 * Bytes of device workspace a solve or adjoint call needs, for `batch` systems of n unknowns
 * (batch = 1 for the single-system calls).  Returns 0 for invalid arguments.
 * Ownership: the caller allocates it (any 256-byte aligned device buffer) and may reuse it
 * across calls; calls sharing one workspace must not overlap on the GPU.
 */
SLA_API size_t sla_cg_workspace_bytes(int64_t n, int64_t batch, int32_t dtype, int32_t precond);

/*
 * Structural check of a CSR matrix (TS Methodology 1: the matrix types the solvers accept).
 * Checks row_ptr bounds and monotonicity, column range, strictly increasing columns within
 * each row and a stored diagonal; with check_symmetric != 0 also that the pattern and values
 * are symmetric (A_ij == A_ji bit for bit).  Synchronises the stream.
 * workspace: device, >= 256 bytes.  Returns SLA_OK or SLA_BAD_CSR; *bad_row (host, may be NULL)
 * receives the first offending row or -1.
 */
SLA_API sla_status sla_validate_csr(const sla_csr *A, int32_t check_symmetric, int64_t *bad_row,
                            void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------- the hot path */

/*
 * y = A x (TS Methodology 1: ".matvec").  x, y: device, n entries of A->dtype; x and y must not
 * overlap.  Each row is summed in storage order with fused multiply-adds.  Asynchronous.
 */
SLA_API sla_status sla_spmv(const sla_csr *A, const void *x, void *y, void *stream);

/*
 * y = A^T x (TS Methodology 1: the backward of an autograd-aware ".matvec" with respect to x).
 * The pattern must be structurally symmetric (every stored (i, j) has a stored (j, i)); values
 * need not be.  Row j of y adds a_ij x_i over the columns i of row j in their order, each a_ij
 * found by a binary search in row i; deterministic.  bad: device uint32 or NULL; a missing partner
 * entry (a pattern that is not structurally symmetric) or an out-of-range index is skipped and
 * sets *bad to 1 (never cleared by the call).  x, y: device, n entries, not overlapping.
 * Asynchronous.
 */
SLA_API sla_status sla_spmv_transpose(const sla_csr *A, const void *x, void *y, uint32_t *bad, void *stream);

/*
 * grad_values[k] = gy[row(k)] * x[col_idx[k]] for every stored entry (TS Methodology 1-2: the
 * gradient of L(A x) with respect to the stored values, for gy = dL/dy, on the pattern only).
 * gy, x: device, n entries; grad_values: device, nnz entries.  Asynchronous.
 */
SLA_API sla_status sla_matvec_grad_values(const sla_csr *A, const void *gy, const void *x, void *grad_values,
                                          void *stream);

/*
 * Solve A x = b by conjugate gradient (TS Methodology 1: the GPU iterative backend; Jacobi
 * preconditioning per TS Significance when opts->precond = SLA_PRECOND_JACOBI).
 *   b        device, n entries.
 *   x0       device, n entries, or NULL for x0 = 0.  May equal x (in-place restart).
 *   x        device, n entries: the solution (the last iterate on every exit).
 *   info     host, or NULL.  With info the call synchronises the stream once and fills it; with
 *            NULL the call is fully asynchronous and the status stays on the device.
 *   history  device, opts->maxit + 1 doubles, or NULL: history[k] = ||r_k|| / ||b|| for
 *            k = 0..iters (entries past iters are not written).
 *   workspace/ws_bytes: device scratch, >= sla_cg_workspace_bytes(n, 1, dtype, precond).
 * The whole iteration runs on the device (opts->loop: one resident kernel, or a CUDA graph whose
 * loop is a device-side conditional); the host does not take part between the first and the
 * last iteration (except with SLA_LOOP_HOST).
 */
SLA_API sla_status sla_cg_solve(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *opts,
                        void *x, sla_cg_info *info, double *history, void *workspace, size_t ws_bytes,
                        void *stream);

/*
 * Adjoint backward of x = A^{-1} b (TS Methodology 2, linear systems): solve A^T lambda = g
 * (A symmetric, so the same CG with the same opts, from lambda = 0), then
 *   grad_b[i]       = lambda[i]                          (written directly: grad_b is lambda)
 *   grad_values[k]  = -lambda[row(k)] * x[col_idx[k]]    (one entry per stored entry, CSR order)
 *   x, g        device, n entries (x: the forward solution; g: dL/dx).
 *   grad_b      device, n entries.  grad_values: device, nnz entries, or NULL to skip.
 *   info        as for sla_cg_solve (status of the adjoint solve).
 */
SLA_API sla_status sla_cg_adjoint(const sla_csr *A, const void *x, const void *g, const sla_cg_opts *opts,
                          void *grad_b, void *grad_values, sla_cg_info *info, void *workspace,
                          size_t ws_bytes, void *stream);

/*
 * grad_values[k] = -lambda[row(k)] * x[col_idx[k]] for every stored entry (TS Methodology 2: the
 * matrix gradient "only on the sparsity pattern").  lambda, x: device, n entries; grad_values:
 * device, nnz entries.  Asynchronous.
 */
SLA_API sla_status sla_grad_values(const sla_csr *A, const void *lambda, const void *x, void *grad_values,
                           void *stream);

/*
 * Batched solve over one shared pattern (TS Methodology 1: one "SparseTensor" holding a shared
 * pattern with a batch of value arrays; "thousands of systems at once").  Each system runs its
 * own CG (own alpha, beta, stopping test); a converged system stops changing.
 *   pattern   CSR whose row_ptr/col_idx are shared; pattern->values is ignored.
 *   values    device, batch x nnz, row-major (system s at values + s*nnz).
 *   b, x0, x  device, batch x n (x0 may be NULL).
 *   info      host, batch entries, or NULL.
 *   history   device, batch x (maxit+1) doubles, or NULL.
 *   workspace >= sla_cg_workspace_bytes(n, batch, dtype, precond).
 */
SLA_API sla_status sla_cg_solve_batched(const sla_csr *pattern, int64_t batch, const void *values, const void *b,
                                const void *x0, const sla_cg_opts *opts, void *x, sla_cg_info *info,
                                double *history, void *workspace, size_t ws_bytes, void *stream);

/*
 * Batched adjoint: for every system s, lambda_s = A_s^{-1} g_s, grad_b[s] = lambda_s,
 * grad_values[s][k] = -lambda_s[row(k)] * x_s[col_idx[k]].  Shapes as in sla_cg_solve_batched;
 * grad_values is batch x nnz (or NULL).
 */
SLA_API sla_status sla_cg_adjoint_batched(const sla_csr *pattern, int64_t batch, const void *values, const void *x,
                                  const void *g, const sla_cg_opts *opts, void *grad_b, void *grad_values,
                                  sla_cg_info *info, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------- general (non-symmetric) A */

/*
 * Bytes of device workspace sla_bicgstab_solve and sla_bicgstab_adjoint need (0 for invalid
 * arguments): eight n-vectors (r, rhat, two p, two v, s, t), the adjoint's A^T (values, column
 * indices and row pointers) with its construction scratch, and the reductions' scratch.
 */
SLA_API size_t sla_bicgstab_workspace_bytes(int64_t n, int64_t nnz, int32_t dtype);

/*
 * BiCGStab solve of a general A x = b (TS Methodology 1: BiCGStab is among the solvers behind
 * .solve; the iteration is the textbook one, van der Vorst, SIAM J. Sci. Stat. Comput. 13, 1992,
 * unpreconditioned): r = b - A x0, rhat = r; per iteration rho = rhat.r, p = r (first) or
 * r + beta (p - omega v) with beta = (rho / rho_prev)(alpha / omega), v = A p,
 * alpha = rho / rhat.v, s = r - alpha v (stop with x += alpha p when ||s|| <= rtol ||b||), t = A s,
 * omega = t.s / t.t, x += alpha p + omega s, r = s - omega t, stop when ||r|| <= rtol ||b||.
 * Zero rhat.v, t.t, omega or rhat.r is SLA_BREAKDOWN (x left at the last iterate).
 * Arguments as for sla_cg_solve, except: opts->precond must be SLA_PRECOND_NONE (else
 * SLA_INVALID_ARG), and opts->loop picks one of two engines.  SLA_LOOP_HOST: three kernels per
 * iteration, the host enqueueing opts->unroll iterations (default 8) between two reads of the
 * device state.  Any other value: the whole solve in one cooperative kernel (one block per SM,
 * three grid barriers per iteration, each wait bounded: an expired wait ends the solve with
 * info->status SLA_TIMEOUT), or the host loop when the cooperative launch cannot be made here.
 * info->path reports the engine that ran (SLA_LOOP_RESIDENT or SLA_LOOP_HOST); info->iters
 * counts iterations (two products with A each).  Dot products are fp64 sums in a fixed order,
 * so an engine gives the same bits run to run.
 */
SLA_API sla_status sla_bicgstab_solve(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *opts,
                                      void *x, sla_cg_info *info, double *history, void *workspace,
                                      size_t ws_bytes, void *stream);

/*
 * Adjoint backward of x = A^{-1} b for a general A (TS Methodology 2): lambda solves
 * A^T lambda = g by the same BiCGStab (same rtol, maxit) from lambda = 0, written into grad_b;
 * then grad_values[e] = -lambda[row(e)] * x[col(e)] on A's pattern (NULL: skipped).  When the
 * pattern is structurally symmetric (a stored (j, i) for every stored (i, j), columns sorted
 * within rows), A^T is used on A's own pattern, every value taken from its partner entry (j, i);
 * otherwise A^T is built explicitly in the workspace (each row's entries in column order, so the
 * result does not depend on the build's atomics; A without duplicate entries).  A malformed row
 * range or column gives info->status SLA_BAD_CSR and nothing is solved.  Arguments and workspace
 * as for sla_bicgstab_solve; x, g, grad_b device n-vectors, grad_values device nnz entries.
 */
SLA_API sla_status sla_bicgstab_adjoint(const sla_csr *A, const void *x, const void *g, const sla_cg_opts *opts,
                                        void *grad_b, void *grad_values, sla_cg_info *info, void *workspace,
                                        size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------- eigenvalue problems */

/* Options of sla_eig_smallest. */
typedef struct sla_eig_opts {
  double tol;           /* stop when ||A v - mu v||_2 <= tol * mu (v of unit norm) */
  int64_t maxit;        /* outer steps (inner CG solves) at most */
  double inner_factor;  /* CG rtol of step k = inner_factor * ||A v_k - mu_k v_k|| / mu_k, in (0, 1) */
  int64_t inner_maxit;  /* CG iterations per solve at most (an unconverged solve still counts as a step) */
  int32_t precond;      /* sla_precond of the inner CG */
  int32_t loop;         /* sla_loop of the inner CG */
} sla_eig_opts;

typedef struct sla_eig_info {
  int64_t iters;        /* outer steps taken (inner solves) */
  int64_t inner_iters;  /* CG iterations over all inner solves */
  double mu;            /* the eigenvalue estimate v^T A v of the returned v */
  double residual;      /* ||A v - mu v||_2 of the returned v */
  int32_t status;       /* SLA_OK, SLA_NOT_CONVERGED (maxit steps), SLA_BREAKDOWN (zero start vector, or
                           v^T A v <= 0: A not positive definite), SLA_NONFINITE, or an inner solve's failure */
  int32_t pad;
} sla_eig_info;

/*
 * Bytes of device workspace sla_eig_smallest needs for n unknowns (0 for invalid arguments):
 * the inner CG's workspace plus two vectors and the step's reduction scratch.
 */
SLA_API size_t sla_eig_workspace_bytes(int64_t n, int32_t dtype, int32_t precond);

/*
 * Smallest eigenpair (mu, v) of a symmetric positive definite A (TS Methodology 1: the ".eigsh"
 * API; the summary names no eigensolver).  Inverse iteration on this library's CG: from the
 * start vector, every step normalises y to v = y / ||y||, forms mu = v^T A v and the residual
 * ||A v - mu v||, and, until the residual is at most tol * mu, solves A y = v by CG started from
 * y = v / mu with the rtol opts->inner_factor * residual / mu (an inexact solve whose accuracy
 * follows the eigen-residual: inexact inverse iteration, Golub and Ye, BIT 40, 2000).
 * Converges for a start vector not orthogonal to the eigenvector, at the rate mu_1 / mu_2 per step.
 *   v          device, n entries of A->dtype: the start vector on entry (not all zero), the unit
 *              eigenvector on return, its sign chosen so that sum_i v_i >= 0.
 *   info       host, required: steps, CG iterations, mu, residual and status.
 *   workspace  device, >= sla_eig_workspace_bytes(n, dtype, opts->precond), 256-byte aligned.
 * The host drives the outer loop (one 48-byte read of the step's scalars per step) and
 * synchronises the stream; the inner solves run on the device as sla_cg_solve does.
 * n = 0 returns SLA_INVALID_ARG (no eigenpair).
 */
SLA_API sla_status sla_eig_smallest(const sla_csr *A, void *v, const sla_eig_opts *opts, sla_eig_info *info,
                                    void *workspace, size_t ws_bytes, void *stream);

/*
 * Bytes of device workspace sla_eigsh needs for k eigenpairs of n unknowns (0 for invalid
 * arguments, k outside 1..16): the inner batched CG's workspace for k systems, three blocks of k
 * vectors and the reductions' scratch.
 */
SLA_API size_t sla_eigsh_workspace_bytes(int64_t n, int64_t k, int32_t dtype, int32_t precond);

/*
 * The k smallest eigenpairs of a symmetric positive definite A, 1 <= k <= min(16, n) (TS
 * Methodology 1: the ".eigsh" API; the summary names no eigensolver).  Block inverse iteration
 * with a Rayleigh-Ritz step (subspace iteration on A^{-1}): the start block is orthonormalised
 * (Cholesky QR, twice); every step forms W = A X and H = X^T W, takes H's eigenvectors Q
 * (theta ascending) to the Ritz vectors X Q and their images W Q, and, until every residual
 * ||A x_s - theta_s x_s|| is at most tol * theta_s, solves A Y = X by CG from Y = X diag(1 / theta)
 * to the rtol inner_factor * max_s residual_s / theta_s, and orthonormalises Y into the next X.
 * When one system fits the resident engine (opts->loop AUTO or RESIDENT) the k solves run there
 * one after another; otherwise together in the batched CG.  The vector s converges at the rate
 * theta_s / theta_{k+1} per step, so a block somewhat larger than the eigenpairs needed converges
 * faster.  Within a
 * multiple eigenvalue the vectors are some orthonormal basis of its eigenspace.
 *   V      device, k x n entries of A->dtype, row-major: the start block on entry (linearly
 *          independent), the unit eigenvectors on return (orthonormal to rounding), each with its
 *          sign chosen so that sum_i v_i >= 0.
 *   mu     host, k doubles: the eigenvalues, ascending (written for SLA_OK and SLA_NOT_CONVERGED).
 *   info   host, required: steps, CG iterations over all vectors, mu = the smallest eigenvalue,
 *          residual = the largest residual, status (SLA_BREAKDOWN also for a rank-deficient block).
 *   workspace device, >= sla_eigsh_workspace_bytes(n, k, dtype, opts->precond), 256-byte aligned.
 * The k x k eigenproblem and Cholesky factor of each step are solved by the host (fp64); the
 * host reads a few k x k results per step and synchronises the stream.
 */
SLA_API sla_status sla_eigsh(const sla_csr *A, int64_t k, void *V, double *mu, const sla_eig_opts *opts,
                             sla_eig_info *info, void *workspace, size_t ws_bytes, void *stream);

/*
 * Eigenvalue gradient on the sparsity pattern (TS Methodology 2, eigenvalue problems:
 * d mu / d A_ij = v_i v_j, Hellmann-Feynman).  For L = sum_s w_s mu_s over k eigenpairs with unit
 * eigenvectors V[s] (s = 0..k-1):
 *   grad_values[e] = sum over s in order of (w_s * V[s][row(e)]) * V[s][col_idx[e]]
 * (the sum starting from the s = 0 term) evaluated in fp64 without fused multiply-adds, then
 * rounded to A->dtype.
 *   k          0..16 (k = 0 writes zeros).
 *   V          device, k x n entries of A->dtype, row-major.
 *   w          host, k doubles, or NULL for all ones.
 *   grad_values device, nnz entries (CSR order).  Asynchronous.
 */
SLA_API sla_status sla_eig_grad_values(const sla_csr *A, int64_t k, const void *V, const double *w,
                                       void *grad_values, void *stream);

/* ---------------------------------------------------------------- distributed row-block CG */

/*
 * One rank's share of a CG solve whose matrix is split into contiguous row blocks, one per rank
 * (TS Methodology 3, "distributed layer with halo exchange": each rank owns a row block, and
 * before its local SpMV receives the values of the vector at the columns it references but does
 * not own).  These calls run one rank's part of each step on its GPU; between them the caller
 * moves halo values between ranks and gathers every rank's partial sums (torch.distributed in the
 * Python layer).  Every rank adds the gathered partials in rank order, so all ranks hold
 * bit-identical scalars and stop at the same iteration.
 *
 * Local block A_ext: the rank's n_own rows with columns renumbered, owned columns 0..n_own-1 first
 * and then the halo columns n_own..n_ext-1 (n_ext = A_ext->n), given as a square CSR of order
 * n_ext whose rows n_own..n_ext-1 are empty.  "own" vectors are device arrays of n_own entries of
 * A_ext->dtype, "ext" vectors n_ext entries (owned values first, then the halo).
 * State: a device buffer of sla_dist_state_bytes() bytes, 256-byte aligned, owned by the caller.
 * Gathered partials: device arrays holding every rank's partials, rank-major ([ranks][k]).
 * Iteration (each call is a no-op once the state's done flag is set, so a caller may enqueue
 * several iterations between two reads of it):
 *   sla_dist_cg_spmv      -> gather 1 partial (p.q)
 *   sla_dist_cg_update    -> gather 2 partials (r.r, r.z)
 *   sla_dist_cg_direction
 *   sla_dist_pack + halo exchange of p
 * The recurrences, stopping rule and status decisions are those of sla_cg_solve; x0 = 0.
 * All calls are asynchronous except sla_dist_cg_info.
 */
SLA_API size_t sla_dist_state_bytes(void);

/*
 * Start of a solve: x = 0, r = b, p = z = M^{-1} r on the owned rows ((Jacobi) dinv = 1 / A_ii);
 * writes this rank's 5 partials (b.b, r.r, r.z, count of non-finite and of non-positive diagonal
 * entries) to `partials` (device, 5 doubles) and resets the state with opts (rtol, maxit, precond;
 * opts->loop and unroll are ignored).  x, r: own vectors; p_ext: ext vector (its halo part is
 * filled by the caller's exchange); z, dinv: own vectors, used only with Jacobi (else may be NULL).
 */
SLA_API sla_status sla_dist_cg_begin(const sla_csr *A_ext, int64_t n_own, const void *b, const sla_cg_opts *opts,
                                     void *x, void *r, void *z, void *p_ext, void *dinv, double *partials,
                                     void *state, void *stream);

/* From the gathered begin partials ([ranks][5]): ||b||, the initial stopping test and status, rho;
 * history (device, maxit+1 doubles, or NULL) receives ||r_0|| / ||b||. */
SLA_API sla_status sla_dist_cg_start(const double *gathered, int32_t ranks, void *state, double *history,
                                     void *stream);

/* q = A_ext p_ext on the owned rows (q: own vector); this rank's partial of p.q into *partial. */
SLA_API sla_status sla_dist_cg_spmv(const sla_csr *A_ext, int64_t n_own, const void *p_ext, void *q, double *partial,
                                    void *state, void *stream);

/* alpha = rho / (p.q summed over the gathered [ranks] partials); x += alpha p; r -= alpha q;
 * z = dinv r (Jacobi); this rank's partials of r.r and r.z into partials[0..1].  p.q <= 0 stops
 * with SLA_BREAKDOWN, a non-finite p.q with SLA_NONFINITE (x left at the last iterate). */
SLA_API sla_status sla_dist_cg_update(int64_t n_own, int32_t dtype, int32_t precond, const double *gathered,
                                      int32_t ranks, void *x, void *r, const void *p_ext, const void *q,
                                      const void *dinv, void *z, double *partials, void *state, void *stream);

/* r.r and r.z summed over the gathered [ranks][2] partials; history[k]; the stopping test
 * (||r|| <= rtol ||b||, maxit, non-finite); else beta = r.z / rho and p = zr + beta p on the owned
 * rows (zr: z with Jacobi, r without). */
SLA_API sla_status sla_dist_cg_direction(int64_t n_own, int32_t dtype, const double *gathered, int32_t ranks,
                                         const void *zr, void *p_ext, double *history, void *state, void *stream);

/* buf[t] = v[idx[t]] for t < m (the owned values a neighbour reads; idx: device int64, entries
 * outside [0, n) give 0).  Asynchronous. */
SLA_API sla_status sla_dist_pack(int64_t n, int32_t dtype, const void *v, const int64_t *idx, int64_t m, void *buf,
                                 void *stream);

/* v[idx[t]] += buf[t] for t < m (TS Methodology 3: the transposed halo exchange of a backward
 * pass, where the values a neighbour computed for this rank's owned entries are added in; idx:
 * device int64, distinct within a call, entries outside [0, n) skipped).  Asynchronous. */
SLA_API sla_status sla_dist_scatter_add(int64_t n, int32_t dtype, void *v, const int64_t *idx, int64_t m,
                                        const void *buf, void *stream);

/* Reads the state (synchronises the stream): iterations, ||r|| / ||b||, status into info (host,
 * may be NULL) and the done flag into *done (host, may be NULL). */
SLA_API sla_status sla_dist_cg_info(const void *state, sla_cg_info *info, int32_t *done, void *stream);

/* ---------------------------------------------------------------- allocation-free variant */

/*
 * sla_cg_solve without a workspace argument, for callers that cannot allocate device memory
 * (plugins inside a host application that owns all device memory, latency-critical paths where
 * an allocation is not allowed, bindings with no device allocator).  The paper has no
 * counterpart: this is a library convenience, not part of the method.
 *   Scratch: a fixed 3,244,544-byte array in the library's own device memory.  CUDA reserves it
 *   on a GPU when it loads the library's device code for this entry point there, which under
 *   CUDA's default lazy module loading is this entry point's first call on that GPU; it is held
 *   until the process exits.  That first call can therefore fail with SLA_CUDA_ERROR when the
 *   GPU has no 3.2 MB left: make it once at start-up.  Systems of up to 65,536 unknowns (one
 *   system, fp32 or fp64, with or without Jacobi) fit; larger n returns SLA_WORKSPACE_TOO_SMALL
 *   before anything is launched.
 *   Set-up: the first call on a device looks up the array's device address on the current
 *   device (cudaGetSymbolAddress) and caches it; make that first call before any stream capture.
 *   Sharing: every call uses the same array.  Each call resets the state it needs, but calls
 *   whose GPU work overlaps (on different streams or threads) race on the array: serialise them.
 *   Allocation: none, neither cudaMalloc/cudaFree nor any allocating library routine; the loop
 *   is driven from the host with plain kernel launches (one 4-byte status read every
 *   opts->unroll iterations; opts->loop is ignored).
 *   Arguments and results as for sla_cg_solve.
 */
SLA_API sla_status sla_cg_solve_static(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *opts,
                                       void *x, sla_cg_info *info, double *history, void *stream);

/* ---------------------------------------------------------------- tuning and testing */

typedef enum sla_spmv_variant {
  SLA_SPMV_PLAIN = 0,  /* default: each thread loads its rows' entries directly */
  SLA_SPMV_TMA = 1     /* the CSR entries of a tile are staged in shared memory by cp.async.bulk with
                          mbarrier double buffering (same per-row arithmetic and results) */
} sla_spmv_variant;

/*
 * Process-wide choice of the SpMV step that the GRAPH and HOST loops launch (not an operation of
 * the method: a tuning switch).  The TMA variant is used only when every array it copies is
 * 16-byte aligned; its mbarrier waits are bounded and fall back to plain loads.  On five-point
 * matrices it measured slower than the plain step, hence the default.  Takes effect at the next
 * solve.  Returns SLA_INVALID_ARG for an unknown variant.
 */
SLA_API sla_status sla_set_spmv_variant(int32_t variant);

/*
 * Introspection of the GRAPH loop's cache (not an operation of the method).  The library keeps up
 * to 32 instantiated graph loops per process, keyed by their shape (value and index types, Jacobi,
 * SpMV variant, launch grid, batch, unroll, device).  A solve of the same shape with other buffers
 * or scalars reuses the cached graph after replacing its kernel nodes' arguments in place; if the
 * runtime refuses that, the entry is rebuilt.  Writes the number of cached graphs, of graphs
 * instantiated and of in-place argument replacements since the process started, to each host
 * pointer that is not NULL.  Always SLA_OK.
 */
SLA_API sla_status sla_graph_cache_stats(int64_t *entries, int64_t *builds, int64_t *updates);

/*
 * Test hook for failure detection (not an operation of the method).  Process-wide bounds of the
 * RESIDENT kernel's grid-barrier wait for the next launches: the barrier waits for `extra`
 * (0 or 1) arrivals beyond its blocks and gives up after `spin_limit` polls (0 = the library
 * default, several seconds; at most 2^26).  With extra = 1 no barrier can complete, so a solve
 * returns SLA_TIMEOUT after spin_limit polls with the CUDA context intact.
 * sla_test_set_barrier_wait(0, 0) restores normal operation.  SLA_INVALID_ARG otherwise.
 */
SLA_API sla_status sla_test_set_barrier_wait(uint32_t extra, int64_t spin_limit);

#ifdef __cplusplus
}
#endif

#endif /* SLA_H_ */
