// Definitions shared by the two on-chip CG engines (the resident kernel of sla_resident.cu and the
// cluster kernel of sla_cluster.cu): the per-iteration scalars and their exact stopping test, the
// device limits they are shaped by, and the per-phase cycle counters of the profiling build.
//
// Method: "torch-sla" technical summary, Methodology 1-2 (Hestenes-Stiefel CG, Jacobi option).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sla_common.cuh"

namespace sla {

#ifdef SLA_PHASE_TIMING
// Profiling build only (compiled out of the library): cycles per phase, summed over iterations,
// for every block: [p-update, spmv, p.q reduce, r-update, r.r reduce, scalars, SM id, iterations].
static __device__ unsigned long long g_phase_cycles[kMaxBlocksPerSystem][8];
#define SLA_PHASE_INIT() unsigned long long ph_[6] = {0, 0, 0, 0, 0, 0}; long long ph_t = clock64()
#define SLA_PHASE(q)                \
  do {                              \
    const long long t_ = clock64(); \
    ph_[q] += t_ - ph_t;            \
    ph_t = t_;                      \
  } while (0)
#define SLA_PHASE_STORE(k)                                                    \
  do {                                                                        \
    if (threadIdx.x == 0) {                                                   \
      unsigned smid_;                                                         \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                      \
      for (int q_ = 0; q_ < 6; ++q_) g_phase_cycles[blockIdx.x][q_] = ph_[q_]; \
      g_phase_cycles[blockIdx.x][6] = smid_;                                  \
      g_phase_cycles[blockIdx.x][7] = (unsigned long long)(k);                \
    }                                                                         \
  } while (0)
#else
#define SLA_PHASE_INIT() \
  do {                   \
  } while (0)
#define SLA_PHASE(q) \
  do {               \
  } while (0)
#define SLA_PHASE_STORE(k) \
  do {                     \
  } while (0)
#endif

// Scalars of the iteration, decided by thread 0 and read by every thread from shared memory
// (fp64 divisions and square roots are far too expensive to repeat in every thread).
struct ResScalars {
  double alpha, beta, alpha_prev, rho, nb;
  double tol, rr_lo, rr_hi;  // stopping test sqrt(r.r) <= tol, decided by comparison outside [lo, hi]
  int go;                    // 1: keep iterating
};

// sqrt(rr) <= tol exactly as the fp64 expression evaluates, without the square root in the common
// case: lo and hi bracket tol^2 with a few ulps of margin (rr <= lo implies sqrt(rr) < tol and
// rr > hi implies sqrt(rr) > tol for correctly rounded sqrt); only rr in between takes the sqrt.
__device__ __forceinline__ bool stop_test(double rr, const ResScalars &S) {
  if (rr <= S.rr_lo) return true;
  if (rr > S.rr_hi) return false;
  return sqrt(rr) <= S.tol;
}

// SM count and opt-in shared memory per block of the current device.
struct ResidentLimits {
  int sms = 0;
  int max_smem = 0;
};

inline ResidentLimits limits() {
  ResidentLimits L;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&L.sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&L.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return L;
}

}  // namespace sla
