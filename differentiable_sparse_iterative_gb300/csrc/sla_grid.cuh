// Grid-wide synchronisation of the persistent (cooperative) kernels: a bounded split-phase grid
// barrier and the deterministic grid totals read after it.  Used by the resident CG and the
// resident BiCGStab; every wait is bounded and raises a timeout flag when it expires, so a
// kernel whose blocks can no longer meet ends with a status instead of spinning.
#pragma once

#include <cuda_runtime.h>

#include "sla_common.cuh"

namespace sla {

// Bounds of the grid barrier's wait.  `extra` arrivals are expected beyond the G blocks: 0 in
// use; a test sets 1 (an arrival that never comes) with a short `limit` to drive the timeout path
// on the GPU and check that the solve returns SLA_TIMEOUT with the context still usable.
struct WaitCfg {
  unsigned extra;
  long long limit;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Split-phase grid barrier over a monotone arrival counter.  grid_arrive: after the block's
// writes (ordered by __syncthreads), thread 0 adds 1 with release semantics (no round trip).
// grid_wait: thread 0 polls with acquire loads until all G blocks of this epoch have arrived, then
// the block synchronises.  The wait is bounded: on expiry (or when another block has timed out) it
// raises the timeout flag and returns false.  Work that needs neither side may run in between.
__device__ __forceinline__ void grid_arrive(unsigned *arrive, unsigned &epoch) {
  __syncthreads();
  ++epoch;
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(arrive), "r"(1u) : "memory");
}

__device__ __forceinline__ bool grid_wait(unsigned *arrive, unsigned *timeout, unsigned G, unsigned epoch,
                                          const WaitCfg &wc) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    const unsigned target = epoch * G + wc.extra;
    int ok = 1;
    long long spins = 0;
    while (ld_acquire(arrive) < target) {
      if (*(volatile unsigned *)timeout) { ok = 0; break; }
      if (++spins > wc.limit) {
        atomicExch(timeout, 1u);
        ok = 0;
        break;
      }
      if (spins > 256) __nanosleep(32);
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ bool grid_barrier(unsigned *arrive, unsigned *timeout, unsigned G, unsigned &epoch,
                                             const WaitCfg &wc) {
  grid_arrive(arrive, epoch);
  return grid_wait(arrive, timeout, G, epoch, wc);
}

// Threads per block of the persistent kernels whose block sums go through block_publish.
constexpr int kPublishBlock = 1024;

// Deterministic all-reduce across the G blocks, in three steps so that the fp64 work on the
// critical path is short:
//  1. block_publish: every thread's value goes through shared memory; warps 0-3 (one per SM
//     sub-partition) each add 256 of them (a depth-3 pairwise tree per lane, then a shuffle
//     tree) and thread 0 adds the four warp sums; the block sum goes to part[j][bid];
//  2. grid_barrier;
//  3. warp_totals (warp 0 only): lane l adds part[j][l], part[j][l+32], ... in order, then a
//     butterfly leaves the identical total in every lane.
// Every block adds the same numbers in the same order, so all blocks hold bit-identical totals.
template <int NV>
__device__ __forceinline__ void block_publish(const double (&v)[NV], double *sbuf, double *part) {
  static_assert(kPublishBlock == 1024, "four warps of 256 values each");
  __shared__ double s4[2][4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int j0 = 0; j0 < NV; j0 += 2) {
    const int nj = (NV - j0) < 2 ? (NV - j0) : 2;
#pragma unroll
    for (int j = 0; j < nj; ++j) sbuf[j * kPublishBlock + tid] = v[j0 + j];
    __syncthreads();
    if (warp < 4) {
#pragma unroll
      for (int j = 0; j < nj; ++j) {
        const double *b = sbuf + j * kPublishBlock + warp * 256 + lane;
        const double a0 = b[0] + b[32], a1 = b[64] + b[96], a2 = b[128] + b[160], a3 = b[192] + b[224];
        const double t = warp_sum((a0 + a1) + (a2 + a3));
        if (lane == 0) s4[j][warp] = t;
      }
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int j = 0; j < nj; ++j)
        part[(size_t)(j0 + j) * kMaxBlocksPerSystem + blockIdx.x] = (s4[j][0] + s4[j][1]) + (s4[j][2] + s4[j][3]);
    }
  }
}

// The wait bounds of the next cooperative launch (0 extra arrivals and the full spin limit unless
// sla_test_set_barrier_wait changed them).
WaitCfg launch_wait_cfg();

__device__ __forceinline__ double warp_allsum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp 0 only: the grid totals, identical in every lane.
template <int NV>
__device__ __forceinline__ void warp_totals(const double *part, int G, double (&tot)[NV]) {
  const int lane = threadIdx.x & 31;
  // all loads of a 256-block slab first (one L2 round trip instead of one per 32 blocks), then a
  // fixed pairwise tree per lane: the order depends only on G, so every block gets the same bits
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const double *pj = part + (size_t)j * kMaxBlocksPerSystem;
    double t = 0.0;
    for (int b0 = 0; b0 < G; b0 += 256) {
      double v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int b = b0 + lane + 32 * u;
        v[u] = b < G ? __ldcg(pj + b) : 0.0;
      }
      t += ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    }
    tot[j] = warp_allsum(t);
  }
}

}  // namespace sla
