// Host-side internals shared by the libsla translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sla.h"

namespace sla {

// Records a CUDA error for sla_last_cuda_error() and returns SLA_CUDA_ERROR.
sla_status fail(cudaError_t e);

// Adds host-side kernel launches to the process-wide count.
void count_launches(uint64_t k);

// The sla_loop the last solve on this thread ran (reported in sla_cg_info.path).
void set_last_path(int path);

// Copies the per-system control blocks back, synchronises the stream and fills info[batch].
struct Ctl;
struct Glob;
sla_status read_info(const Ctl *ctl, const Glob *glob, int64_t batch, cudaStream_t stream, sla_cg_info *info);

// Device-resident CG for `batch` systems sharing A's pattern (values at values + s*val_stride).
sla_status cg_entry(const sla_csr *A, int64_t batch, const void *values, int64_t val_stride, const void *b,
                    const void *x0, const sla_cg_opts *o, void *x, sla_cg_info *info, double *history, void *ws,
                    cudaStream_t st,
                    bool halo_ws = true);

size_t workspace_bytes(int64_t n, int64_t batch, int dtype, int precond);

// True when one system of n unknowns fits the resident (shared-memory) CG kernel on this device.
bool resident_fits(int64_t n, int64_t batch, int dtype, int precond, int64_t maxit);

// True when every system of a batch fits one thread-block cluster (cluster-resident CG kernel).
bool cluster_fits(int64_t n, int64_t batch, int dtype, int precond);

// Argument checks of the entry points (no CUDA call): p aligned to a bytes; a CSR descriptor
// (sizes, types, non-NULL arrays, alignment; values too when need_values); a vector of A's
// dtype (NULL allowed when allow_null or n == 0).
bool aligned(const void *p, size_t a);
sla_status check_csr(const sla_csr *A, bool need_values);
sla_status check_vec(const void *p, const sla_csr *A, bool allow_null);
sla_status check_opts(const sla_cg_opts *o);

#define SLA_CHECK(expr)            \
  do {                             \
    sla_status st_ = (expr);       \
    if (st_ != SLA_OK) return st_; \
  } while (0)

// grad_values[s][k] = -lambda_s[row(k)] * x_s[col(k)] for `batch` systems (asynchronous).
sla_status grad_values_entry(const sla_csr *A, int64_t batch, const void *lambda, const void *x, void *gv,
                             cudaStream_t st);

}  // namespace sla
