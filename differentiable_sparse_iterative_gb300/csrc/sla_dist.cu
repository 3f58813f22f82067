// One rank's share of the distributed row-block CG ("torch-sla" technical summary, Methodology 3:
// distributed layer with halo exchange; Methodology 1-2 for the CG itself and its adjoint).
//
// The global matrix is split into contiguous row blocks, one per rank.  A rank holds its rows
// with the columns renumbered: owned columns 0..n_own-1, then the halo columns it references but
// does not own, n_own..n_ext-1.  The library sees that block as a square CSR of order n_ext whose
// rows n_own..n_ext-1 are empty, so the ordinary CSR checks and the pattern gradient apply to it
// unchanged.  Between the calls below, the caller (the Python layer over torch.distributed) moves
// the halo values of p (and of x for the gradient) and gathers every rank's partial sums; each
// rank then adds the gathered partials in rank order, so every rank holds bit-identical scalars
// and takes the same decisions, and no rank can stop while another goes on.
//
// Per iteration (textbook Hestenes-Stiefel CG, as the single-GPU engines):
//   spmv:      q = A_loc p_ext on the owned rows; partial of p.q           -> gather
//   update:    alpha = rho / sum(p.q); x += alpha p; r -= alpha q; z = M^-1 r; partials of r.r, r.z
//                                                                          -> gather
//   direction: rr = sum(r.r); stopping test; beta = sum(r.z) / rho; p = z + beta p
//   pack:      the owned values of p that the neighbours read               -> halo exchange
// A device-side done flag makes every call after the stop a no-op, so the host may enqueue
// several iterations between two reads of it.
#include <cuda_runtime.h>

#include <cmath>

#include "sla_common.cuh"
#include "sla_host.h"

namespace sla {

namespace {

constexpr int kDistSlots = 5;  // partial-sum rows of one rank's reductions (the begin step has 5 sums)

struct DistState {
  double rho;       // r.z (r.r without preconditioner) of the current iterate
  double alpha;     // step length of the last update
  double beta;      // beta of the last direction update
  double nb;        // ||b||_2 over all ranks
  double tol;       // rtol * ||b||
  double rtol;
  double rel_res;   // ||r|| / ||b|| at the latest residual
  int64_t k;        // completed iterations
  int64_t maxit;
  int32_t status;
  int32_t done;     // 1 once the solve has stopped (every later call is a no-op)
  int32_t precond;
  uint32_t ticket;  // arrival counter of the last-block reductions
  uint32_t bad_csr;
  uint32_t pad;
  double part[kDistSlots][kMaxBlocksPerSystem];
};

// True in the block that arrives last at this point of the kernel (every other block has passed
// everything it did before).  Thread 0 of that block may then update the state's scalars.
__device__ __forceinline__ bool arrive_last(DistState *S) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned t = atomicAdd(&S->ticket, 1u);
    s_last = (t == gridDim.x - 1);
    if (s_last) S->ticket = 0u;
  }
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  return true;
}

int dist_grid(int64_t n_own) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (n_own + kBlock * 4 - 1) / (kBlock * 4);
  const int64_t cap = (int64_t)sms * 8 < kMaxBlocksPerSystem ? (int64_t)sms * 8 : kMaxBlocksPerSystem;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

// Sum of R gathered values, stride `stride`, in rank order (every rank gets the same bits).
__device__ __forceinline__ double rank_sum(const double *g, int R, int stride, int j) {
  double s = 0.0;
  for (int q = 0; q < R; ++q) s += g[(size_t)q * stride + j];
  return s;
}

// Publishes NV block sums (valid in thread 0); in the last block, reduces them in a fixed order
// into out[0..NV) and returns true there.
template <int NV>
__device__ __forceinline__ bool dist_reduce(double (&v)[NV], DistState *S, double *out) {
  block_sum<NV>(v);
  __shared__ int s_last;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int j = 0; j < NV; ++j) S->part[j][blockIdx.x] = v[j];
    __threadfence();
    const unsigned t = atomicAdd(&S->ticket, 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  if (threadIdx.x < 32) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double t = 0.0;
      for (int i = threadIdx.x; i < (int)gridDim.x; i += 32) t += __ldcg(&S->part[j][i]);
      t = warp_sum(t);
      if (threadIdx.x == 0) out[j] = t;
    }
  }
  if (threadIdx.x == 0) S->ticket = 0u;
  return true;
}

// x = 0, r = b, (Jacobi) dinv = 1/A_ii and z = dinv r, p = z; partials b.b, r.r, r.z and the counts
// of non-finite and non-positive diagonal entries.
template <typename V, typename I, bool JAC>
__global__ void __launch_bounds__(kBlock) dist_begin_kernel(int64_t n_own, int64_t nnz, const I *__restrict__ rp,
                                                            const int32_t *__restrict__ ci,
                                                            const V *__restrict__ val, const V *__restrict__ b,
                                                            V *__restrict__ x, V *__restrict__ r, V *__restrict__ z,
                                                            V *__restrict__ p, V *__restrict__ dinv, double *out,
                                                            DistState *S) {
  double acc[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n_own; i += (int64_t)gridDim.x * kBlock) {
    const V bi = b[i];
    x[i] = V(0);
    r[i] = bi;
    acc[0] = fma((double)bi, (double)bi, acc[0]);
    acc[1] = fma((double)bi, (double)bi, acc[1]);
    V zi = bi;
    if (JAC) {
      int64_t e0, e1;
      row_range(rp, i, nnz, e0, e1, &S->bad_csr);
      V d = V(0);
      for (int64_t e = e0; e < e1; ++e)
        if (ci[e] == (int32_t)i) d = val[e];
      if (!isfinite((double)d)) acc[3] += 1.0;
      else if (!(d > V(0))) acc[4] += 1.0;
      const V di = V(1) / d;
      dinv[i] = di;
      zi = di * bi;
      z[i] = zi;
      acc[2] = fma((double)bi, (double)zi, acc[2]);
    }
    p[i] = zi;
  }
  dist_reduce<5>(acc, S, out);
}

// From the gathered begin partials [R][5]: ||b||, the initial residual test, rho; history[0].
__global__ void dist_start_kernel(const double *g, int R, DistState *S, double *history) {
  if (threadIdx.x != 0) return;
  const double bb = rank_sum(g, R, 5, 0), rr = rank_sum(g, R, 5, 1), rz = rank_sum(g, R, 5, 2);
  const double nonfinite = rank_sum(g, R, 5, 3), nonpos = rank_sum(g, R, 5, 4);
  const double nb = sqrt(bb);
  const bool jac = S->precond == SLA_PRECOND_JACOBI;
  S->nb = nb;
  S->k = 0;
  S->alpha = S->beta = 0.0;
  S->rel_res = 0.0;
  int status = SLA_NOT_CONVERGED, done = 1;
  if (!isfinite(nb)) {
    status = SLA_NONFINITE;
  } else if (nb == 0.0) {
    status = SLA_OK;
    if (history) history[0] = 0.0;
  } else if (jac && nonfinite > 0.0) {
    status = SLA_NONFINITE;
  } else if (jac && nonpos > 0.0) {
    status = SLA_BREAKDOWN;
  } else {
    S->rel_res = sqrt(rr) / nb;
    if (history) history[0] = S->rel_res;
    if (!isfinite(rr)) status = SLA_NONFINITE;
    else if (sqrt(rr) <= S->rtol * nb) status = SLA_OK;
    else if (S->maxit == 0) status = SLA_NOT_CONVERGED;
    else {
      done = 0;
      S->rho = jac ? rz : rr;
      S->tol = S->rtol * nb;
    }
  }
  S->status = status;
  S->done = done;
}

// q = A_loc p_ext on the owned rows; partial of p.q.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) dist_spmv_kernel(int64_t n_own, int64_t n_ext, int64_t nnz,
                                                           const I *__restrict__ rp, const int32_t *__restrict__ ci,
                                                           const V *__restrict__ val, const V *__restrict__ p,
                                                           V *__restrict__ q, double *out, DistState *S) {
  if (S->done) return;  // written only by earlier kernels: the same in every block
  double acc[1] = {0.0};
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n_own; i += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, i, nnz, e0, e1, &S->bad_csr);
    V s = V(0);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t c = ci[e];
      if (col_ok(c, (int32_t)n_ext, &S->bad_csr)) s = fmav<V>(val[e], p[c], s);
    }
    q[i] = s;
    acc[0] = fma((double)p[i], (double)s, acc[0]);
  }
  dist_reduce<1>(acc, S, out);
}

// alpha = rho / (p.q summed over ranks); x += alpha p; r -= alpha q; z = dinv r; partials r.r, r.z.
template <typename V, bool JAC>
__global__ void __launch_bounds__(kBlock) dist_update_kernel(int64_t n_own, const double *g, int R,
                                                             V *__restrict__ x, V *__restrict__ r,
                                                             const V *__restrict__ p, const V *__restrict__ q,
                                                             const V *__restrict__ dinv, V *__restrict__ z,
                                                             double *out, DistState *S) {
  if (S->done) return;
  __shared__ double s_alpha;
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    const double pq = rank_sum(g, R, 1, 0);
    s_bad = !isfinite(pq) ? SLA_NONFINITE : (!(pq > 0.0) ? SLA_BREAKDOWN : 0);
    s_alpha = s_bad ? 0.0 : S->rho / pq;
  }
  __syncthreads();
  const int bad = s_bad;
  const V va = (V)s_alpha;
  double acc[2] = {0.0, 0.0};
  if (!bad) {
    for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n_own; i += (int64_t)gridDim.x * kBlock) {
      x[i] = fmav<V>(va, p[i], x[i]);
      const V ri = fmav<V>(-va, q[i], r[i]);
      r[i] = ri;
      acc[0] = fma((double)ri, (double)ri, acc[0]);
      if (JAC) {
        const V zi = dinv[i] * ri;
        z[i] = zi;
        acc[1] = fma((double)ri, (double)zi, acc[1]);
      }
    }
  }
  if (dist_reduce<2>(acc, S, out) && threadIdx.x == 0) {
    S->alpha = s_alpha;
    if (bad) {
      S->status = bad;
      S->done = 1;
    }
  }
}

// rr, rz summed over ranks; history; stopping test; beta = rz / rho; p = z + beta p.
template <typename V>
__global__ void __launch_bounds__(kBlock) dist_direction_kernel(int64_t n_own, const double *g, int R,
                                                                const V *__restrict__ zr, V *__restrict__ p,
                                                                double *history, DistState *S) {
  if (S->done) return;
  __shared__ double s_beta, s_rz;
  __shared__ int s_stop;
  if (threadIdx.x == 0) {
    const double rr = rank_sum(g, R, 2, 0);
    const double rz = S->precond == SLA_PRECOND_JACOBI ? rank_sum(g, R, 2, 1) : rr;
    const int64_t k = S->k + 1;
    int stop = 0;
    if (!isfinite(rr)) stop = SLA_NONFINITE + 16;
    else if (sqrt(rr) <= S->tol) stop = SLA_OK + 16;
    else if (k >= S->maxit) stop = SLA_NOT_CONVERGED + 16;
    s_stop = stop;
    s_rz = rz;
    s_beta = rz / S->rho;
    if (blockIdx.x == 0) {
      const double rel = sqrt(rr) / S->nb;
      if (history) history[k] = rel;
    }
  }
  __syncthreads();
  if (!s_stop) {
    const V vb = (V)s_beta;
    for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n_own; i += (int64_t)gridDim.x * kBlock)
      p[i] = fmav<V>(vb, p[i], zr[i]);
  }
  // every block has read rho, k and tol above; the last block to arrive updates them
  if (arrive_last(S) && threadIdx.x == 0) {
    const double rr = rank_sum(g, R, 2, 0);
    S->k += 1;
    S->rel_res = sqrt(rr) / S->nb;
    if (s_stop) {
      S->status = s_stop - 16;
      S->done = 1;
    } else {
      S->beta = s_beta;
      S->rho = s_rz;
    }
  }
}

// buf[t] = v[idx[t]] (the owned values a neighbour reads).
template <typename V>
__global__ void __launch_bounds__(kBlock) dist_pack_kernel(int64_t n, const V *__restrict__ v,
                                                           const int64_t *__restrict__ idx, int64_t m,
                                                           V *__restrict__ buf) {
  for (int64_t t = blockIdx.x * (int64_t)kBlock + threadIdx.x; t < m; t += (int64_t)gridDim.x * kBlock) {
    const int64_t i = idx[t];
    buf[t] = (uint64_t)i < (uint64_t)n ? v[i] : V(0);
  }
}

// v[idx[t]] += buf[t] (the contributions a neighbour computed for this rank's owned entries; the
// indices of one call are distinct, so the adds do not race).
template <typename V>
__global__ void __launch_bounds__(kBlock) dist_scatter_add_kernel(int64_t n, V *__restrict__ v,
                                                                  const int64_t *__restrict__ idx, int64_t m,
                                                                  const V *__restrict__ buf) {
  for (int64_t t = blockIdx.x * (int64_t)kBlock + threadIdx.x; t < m; t += (int64_t)gridDim.x * kBlock) {
    const int64_t i = idx[t];
    if ((uint64_t)i < (uint64_t)n) v[i] += buf[t];
  }
}

sla_status launched() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  return SLA_OK;
}

sla_status check_state(const void *state) {
  return (state && aligned(state, 256)) ? SLA_OK : SLA_INVALID_ARG;
}

template <typename V, typename I>
sla_status begin_t(const sla_csr *A, int64_t n_own, const void *b, void *x, void *r, void *z, void *p, void *dinv,
                   double *out, DistState *S, bool jac, cudaStream_t st) {
  const int G = dist_grid(n_own);
  if (jac)
    dist_begin_kernel<V, I, true><<<G, kBlock, 0, st>>>(n_own, A->nnz, (const I *)A->row_ptr, A->col_idx,
                                                        (const V *)A->values, (const V *)b, (V *)x, (V *)r, (V *)z,
                                                        (V *)p, (V *)dinv, out, S);
  else
    dist_begin_kernel<V, I, false><<<G, kBlock, 0, st>>>(n_own, A->nnz, (const I *)A->row_ptr, A->col_idx,
                                                         (const V *)A->values, (const V *)b, (V *)x, (V *)r,
                                                         nullptr, (V *)p, nullptr, out, S);
  return launched();
}

template <typename V, typename I>
sla_status spmv_t(const sla_csr *A, int64_t n_own, const void *p, void *q, double *out, DistState *S,
                  cudaStream_t st) {
  dist_spmv_kernel<V, I><<<dist_grid(n_own), kBlock, 0, st>>>(n_own, A->n, A->nnz, (const I *)A->row_ptr,
                                                              A->col_idx, (const V *)A->values, (const V *)p,
                                                              (V *)q, out, S);
  return launched();
}

}  // namespace
}  // namespace sla

using namespace sla;

extern "C" {

size_t sla_dist_state_bytes(void) { return align256(sizeof(DistState)); }

sla_status sla_dist_cg_begin(const sla_csr *A_ext, int64_t n_own, const void *b, const sla_cg_opts *opts, void *x,
                             void *r, void *z, void *p_ext, void *dinv, double *partials, void *state,
                             void *stream) {
  SLA_CHECK(check_csr(A_ext, true));
  SLA_CHECK(check_opts(opts));
  SLA_CHECK(check_state(state));
  if (n_own < 0 || n_own > A_ext->n || !partials) return SLA_INVALID_ARG;
  const bool jac = opts->precond == SLA_PRECOND_JACOBI;
  SLA_CHECK(check_vec(b, A_ext, false));
  SLA_CHECK(check_vec(x, A_ext, false));
  SLA_CHECK(check_vec(r, A_ext, false));
  SLA_CHECK(check_vec(p_ext, A_ext, false));
  if (jac) {
    SLA_CHECK(check_vec(z, A_ext, false));
    SLA_CHECK(check_vec(dinv, A_ext, false));
  }
  if (!aligned(partials, 8)) return SLA_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  DistState *S = (DistState *)state;
  DistState init{};
  init.rtol = opts->rtol;
  init.maxit = opts->maxit;
  init.precond = opts->precond;
  init.done = 1;
  init.status = SLA_NOT_CONVERGED;
  // the scalar head of the state (everything before the partial sums) is set from the host
  cudaError_t e = cudaMemcpyAsync(S, &init, offsetof(DistState, part), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(e);
  if (n_own == 0) {
    e = cudaMemsetAsync(partials, 0, 5 * sizeof(double), st);
    return e == cudaSuccess ? SLA_OK : fail(e);
  }
  if (A_ext->dtype == SLA_F64) {
    if (A_ext->rowptr_type == SLA_I64)
      return begin_t<double, int64_t>(A_ext, n_own, b, x, r, z, p_ext, dinv, partials, S, jac, st);
    return begin_t<double, int32_t>(A_ext, n_own, b, x, r, z, p_ext, dinv, partials, S, jac, st);
  }
  if (A_ext->rowptr_type == SLA_I64)
    return begin_t<float, int64_t>(A_ext, n_own, b, x, r, z, p_ext, dinv, partials, S, jac, st);
  return begin_t<float, int32_t>(A_ext, n_own, b, x, r, z, p_ext, dinv, partials, S, jac, st);
}

sla_status sla_dist_cg_start(const double *gathered, int32_t ranks, void *state, double *history, void *stream) {
  SLA_CHECK(check_state(state));
  if (!gathered || ranks < 1 || !aligned(gathered, 8) || !aligned(history, 8)) return SLA_INVALID_ARG;
  dist_start_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(gathered, ranks, (DistState *)state, history);
  return launched();
}

sla_status sla_dist_cg_spmv(const sla_csr *A_ext, int64_t n_own, const void *p_ext, void *q, double *partial,
                            void *state, void *stream) {
  SLA_CHECK(check_csr(A_ext, true));
  SLA_CHECK(check_state(state));
  if (n_own < 0 || n_own > A_ext->n || !partial || !aligned(partial, 8)) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(p_ext, A_ext, false));
  SLA_CHECK(check_vec(q, A_ext, false));
  cudaStream_t st = (cudaStream_t)stream;
  DistState *S = (DistState *)state;
  if (n_own == 0) {
    const cudaError_t e = cudaMemsetAsync(partial, 0, sizeof(double), st);
    return e == cudaSuccess ? SLA_OK : fail(e);
  }
  if (A_ext->dtype == SLA_F64) {
    if (A_ext->rowptr_type == SLA_I64) return spmv_t<double, int64_t>(A_ext, n_own, p_ext, q, partial, S, st);
    return spmv_t<double, int32_t>(A_ext, n_own, p_ext, q, partial, S, st);
  }
  if (A_ext->rowptr_type == SLA_I64) return spmv_t<float, int64_t>(A_ext, n_own, p_ext, q, partial, S, st);
  return spmv_t<float, int32_t>(A_ext, n_own, p_ext, q, partial, S, st);
}

sla_status sla_dist_cg_update(int64_t n_own, int32_t dtype, int32_t precond, const double *gathered, int32_t ranks,
                              void *x, void *r, const void *p_ext, const void *q, const void *dinv, void *z,
                              double *partials, void *state, void *stream) {
  SLA_CHECK(check_state(state));
  if (n_own < 0 || ranks < 1 || !gathered || !partials || !aligned(partials, 8)) return SLA_INVALID_ARG;
  if (dtype != SLA_F32 && dtype != SLA_F64) return SLA_INVALID_ARG;
  if (precond != SLA_PRECOND_NONE && precond != SLA_PRECOND_JACOBI) return SLA_INVALID_ARG;
  const bool jac = precond == SLA_PRECOND_JACOBI;
  const size_t vs = dtype == SLA_F64 ? 8 : 4;
  if (n_own > 0 && (!x || !r || !p_ext || !q || (jac && (!dinv || !z)))) return SLA_INVALID_ARG;
  if (!aligned(x, vs) || !aligned(r, vs) || !aligned(p_ext, vs) || !aligned(q, vs) || !aligned(dinv, vs) ||
      !aligned(z, vs))
    return SLA_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  DistState *S = (DistState *)state;
  const int G = dist_grid(n_own);
  if (dtype == SLA_F64) {
    if (jac)
      dist_update_kernel<double, true><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (double *)x, (double *)r,
                                                             (const double *)p_ext, (const double *)q,
                                                             (const double *)dinv, (double *)z, partials, S);
    else
      dist_update_kernel<double, false><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (double *)x, (double *)r,
                                                              (const double *)p_ext, (const double *)q, nullptr,
                                                              nullptr, partials, S);
  } else {
    if (jac)
      dist_update_kernel<float, true><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (float *)x, (float *)r,
                                                            (const float *)p_ext, (const float *)q,
                                                            (const float *)dinv, (float *)z, partials, S);
    else
      dist_update_kernel<float, false><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (float *)x, (float *)r,
                                                             (const float *)p_ext, (const float *)q, nullptr,
                                                             nullptr, partials, S);
  }
  return launched();
}

sla_status sla_dist_cg_direction(int64_t n_own, int32_t dtype, const double *gathered, int32_t ranks,
                                 const void *zr, void *p_ext, double *history, void *state, void *stream) {
  SLA_CHECK(check_state(state));
  if (n_own < 0 || ranks < 1 || !gathered) return SLA_INVALID_ARG;
  if (dtype != SLA_F32 && dtype != SLA_F64) return SLA_INVALID_ARG;
  const size_t vs = dtype == SLA_F64 ? 8 : 4;
  if (n_own > 0 && (!zr || !p_ext)) return SLA_INVALID_ARG;
  if (!aligned(zr, vs) || !aligned(p_ext, vs) || !aligned(history, 8)) return SLA_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  DistState *S = (DistState *)state;
  const int G = dist_grid(n_own);
  if (dtype == SLA_F64)
    dist_direction_kernel<double><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (const double *)zr,
                                                        (double *)p_ext, history, S);
  else
    dist_direction_kernel<float><<<G, kBlock, 0, st>>>(n_own, gathered, ranks, (const float *)zr, (float *)p_ext,
                                                       history, S);
  return launched();
}

sla_status sla_dist_pack(int64_t n, int32_t dtype, const void *v, const int64_t *idx, int64_t m, void *buf,
                         void *stream) {
  if (n < 0 || m < 0 || (dtype != SLA_F32 && dtype != SLA_F64)) return SLA_INVALID_ARG;
  if (m == 0) return SLA_OK;
  const size_t vs = dtype == SLA_F64 ? 8 : 4;
  if (!v || !idx || !buf || !aligned(v, vs) || !aligned(idx, 8) || !aligned(buf, vs)) return SLA_INVALID_ARG;
  const int G = dist_grid(m);
  if (dtype == SLA_F64)
    dist_pack_kernel<double><<<G, kBlock, 0, (cudaStream_t)stream>>>(n, (const double *)v, idx, m, (double *)buf);
  else
    dist_pack_kernel<float><<<G, kBlock, 0, (cudaStream_t)stream>>>(n, (const float *)v, idx, m, (float *)buf);
  return launched();
}

sla_status sla_dist_scatter_add(int64_t n, int32_t dtype, void *v, const int64_t *idx, int64_t m, const void *buf,
                                void *stream) {
  if (n < 0 || m < 0 || (dtype != SLA_F32 && dtype != SLA_F64)) return SLA_INVALID_ARG;
  if (m == 0) return SLA_OK;
  const size_t vs = dtype == SLA_F64 ? 8 : 4;
  if (!v || !idx || !buf || !aligned(v, vs) || !aligned(idx, 8) || !aligned(buf, vs)) return SLA_INVALID_ARG;
  const int G = dist_grid(m);
  if (dtype == SLA_F64)
    dist_scatter_add_kernel<double><<<G, kBlock, 0, (cudaStream_t)stream>>>(n, (double *)v, idx, m,
                                                                            (const double *)buf);
  else
    dist_scatter_add_kernel<float><<<G, kBlock, 0, (cudaStream_t)stream>>>(n, (float *)v, idx, m,
                                                                           (const float *)buf);
  return launched();
}

sla_status sla_dist_cg_info(const void *state, sla_cg_info *info, int32_t *done, void *stream) {
  SLA_CHECK(check_state(state));
  if (!info && !done) return SLA_INVALID_ARG;
  DistState h;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&h, state, offsetof(DistState, part), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(e);
  if (done) *done = h.done;
  if (info) {
    info->iters = h.k;
    info->rel_res = h.rel_res;
    info->status = h.bad_csr ? SLA_BAD_CSR : h.status;
    info->path = SLA_LOOP_HOST;
    info->kernels = 0;
  }
  return SLA_OK;
}

}  // extern "C"
