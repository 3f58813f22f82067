// Shared device-side definitions of libsla: control block, workspace layout,
// deterministic reductions and the "last block reduces" protocol.
//
// The library solves the CSR systems of "torch-sla: Differentiable Sparse
// Linear Algebra with Adjoint Solvers and Sparse Tensor Parallelism for
// PyTorch" (Chi, Wen), technical summary, Methodology 1-2, on one GB300.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sla.h"

namespace sla {

constexpr int kBlock = 256;                  // threads per block of every row kernel
constexpr int kWarps = kBlock / 32;
constexpr int kMaxBlocksPerSystem = 2048;    // partial-sum slots per system and reduction
constexpr int kRedSlots = 6;                 // partial-sum rows: 5 (setup / r.r, r.z) + 1 (p.q, resident kernel)

// Per-system solver state, resident on the device for the whole solve.
struct Ctl {
  double rho;        // r.z of the current iterate
  double alpha;      // step length of the current (or last) iteration
  double beta;       // beta of the last completed iteration
  double nb;         // ||b||_2
  double rel_res;    // ||r|| / ||b|| of the latest residual
  int64_t k;         // completed iterations
  int32_t status;    // sla_status
  int32_t done;      // 1 once this system has stopped
  int32_t pending;   // 0: nothing; 1: x += alpha * p[last_parity] at finish; 2: x = 0 at finish
  int32_t last_parity;
  uint32_t ticket;   // arrival counter of the last-block reduction (returns to 0 after each use)
  uint32_t pad;
};
static_assert(sizeof(Ctl) % 8 == 0, "Ctl must stay 8-byte aligned");

// Whole-call state.
struct Glob {
  uint32_t active;                // systems still iterating
  uint32_t bodies;                // loop bodies executed
  unsigned long long kernels;     // kernel executions of this call
  uint32_t safety_stop;           // 1 if the loop was cut by the body bound (never expected)
  uint32_t bad_csr;               // 1 if a row range or column index was out of bounds (entry skipped)
  uint32_t barrier;               // arrival counter of the resident kernel's grid barrier
  uint32_t timeout;               // 1 if a bounded grid-barrier wait expired
};

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout (offsets in bytes from the workspace base).
struct Layout {
  size_t glob, ctl, partials, r, p0, p1, q, dinv, z, halo, total;
};

// halo: one bit per row (shared by the systems of a batch), set for the rows that another block of
// the resident kernel reads; last, so that a layout without it keeps every other offset.
__host__ __device__ constexpr Layout make_layout(int64_t n, int64_t batch, size_t vbytes, bool jacobi,
                                                 bool with_halo = true) {
  Layout L{};
  size_t off = 0;
  L.glob = off; off += align256(sizeof(Glob));
  L.ctl = off; off += align256(sizeof(Ctl) * (size_t)batch);
  L.partials = off; off += align256(sizeof(double) * (size_t)kRedSlots * kMaxBlocksPerSystem * (size_t)batch);
  size_t vec = align256(vbytes * (size_t)n * (size_t)batch);
  L.r = off; off += vec;
  L.p0 = off; off += vec;
  L.p1 = off; off += vec;
  L.q = off; off += vec;
  L.dinv = off; off += jacobi ? vec : 0;
  L.z = off; off += jacobi ? vec : 0;  // z = M^{-1} r, kept so the SpMV step reads one vector
  L.halo = off; off += with_halo ? align256(sizeof(uint32_t) * (size_t)((n + 31) / 32)) : 0;
  L.total = off;
  return L;
}

// Everything a solve kernel needs, passed by value (it lives in the kernel's parameter bank).
template <typename V, typename I>
struct Prob {
  const I *rp;
  const int32_t *ci;
  const V *val;          // values of system 0
  const V *b;            // right-hand side of system 0
  const V *x0;           // NULL: start from 0
  V *x;                  // solution of system 0
  V *r;
  V *p[2];               // ping-pong search directions
  V *q;
  V *dinv;               // Jacobi: 1 / A_ii
  V *z;                  // Jacobi: z = dinv * r (written with r; the SpMV step reads z, not r and dinv)
  double *partials;      // [batch][kRedSlots][kMaxBlocksPerSystem]
  Ctl *ctl;              // [batch]
  Glob *glob;
  double *history;       // [batch][maxit+1] or NULL
  int64_t val_stride;    // nnz for batched values, 0 when all systems share one value array
  int64_t nnz;
  int64_t maxit;
  double rtol;
  uint32_t *halo;        // row bitmap of the resident kernel, or NULL (then every row is published)
  int32_t n;
  int32_t G;             // blocks per system
  int32_t batch;
  int32_t pad;
};

template <typename V> __device__ __forceinline__ V fmav(V a, V b, V c);
template <> __device__ __forceinline__ double fmav<double>(double a, double b, double c) { return fma(a, b, c); }
template <> __device__ __forceinline__ float fmav<float>(float a, float b, float c) { return fmaf(a, b, c); }

// Rows [c0, c1) of block bx out of G equal contiguous chunks.
__device__ __forceinline__ void chunk_of(int64_t n, int G, int bx, int64_t &c0, int64_t &c1) {
  c0 = n * bx / G;
  c1 = n * (bx + 1) / G;
}

// As chunk_of, with every chunk boundary but the end rounded down to a multiple of `align` rows
// (64-bit throughout), so that only the last block has a ragged tail.
__device__ __forceinline__ void chunk_aligned(int64_t n, int G, int bx, int64_t align, int64_t &c0, int64_t &c1) {
  c0 = (n * bx / G) / align * align;
  c1 = bx + 1 == G ? n : (n * (bx + 1) / G) / align * align;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum of NV values per thread of a BLOCK-thread block, in a fixed order; the result
// is in thread 0.  fp64 instructions are the scarce resource on this GPU (2 FMA per SM per clock,
// so one 32-lane fp64 instruction holds an SM sub-partition for 64 cycles): instead of a shuffle
// tree in every warp, the values go through shared memory and warp 0 alone adds them, lane l
// summing entries l, l+32, ... in order, then a 5-step shuffle tree.  That is BLOCK/32 + 4
// fp64 warp-instructions per value instead of 5 * BLOCK/32 + 5.
template <int NV, int BLOCK>
__device__ __forceinline__ void block_sum_n(double (&v)[NV]) {
  static_assert(BLOCK % 32 == 0, "block size must be a multiple of 32");
  __shared__ double sbuf[NV][BLOCK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < NV; ++j) sbuf[j][threadIdx.x] = v[j];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double t = sbuf[j][lane];
#pragma unroll
      for (int k = 1; k < BLOCK / 32; ++k) t += sbuf[j][lane + 32 * k];
      v[j] = warp_sum(t);
    }
  }
  __syncthreads();
}

template <int NV>
__device__ __forceinline__ void block_sum(double (&v)[NV]) {
  block_sum_n<NV, kBlock>(v);
}

// Publishes this block's sums (valid in thread 0) as partials[j][bx] and returns true in the
// block that arrives last.  The last block then reads all G partials with reduce_partials().
template <int NV>
__device__ __forceinline__ bool publish_last(const double (&v)[NV], double *part, uint32_t *ticket, int G,
                                             int bx) {
  __shared__ int s_last;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int j = 0; j < NV; ++j) part[(size_t)j * kMaxBlocksPerSystem + bx] = v[j];
    __threadfence();
    unsigned t = atomicAdd(ticket, 1u);
    s_last = (t == (unsigned)(G - 1));
  }
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  return true;
}

// Sum of the G partials of each reduction in a fixed order: thread t adds slots t, t+kBlock, ...
// in that order, then block_sum.  Independent of which block came last.  Result in thread 0;
// the ticket is returned to 0 for the next kernel.
template <int NV>
__device__ __forceinline__ void reduce_partials(const double *part, int G, uint32_t *ticket, double (&tot)[NV]) {
  // warp 0 alone: lane l adds partials l, l+32, ... in order, then the shuffle tree
  if (threadIdx.x < 32) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double t = 0.0;
      for (int i = threadIdx.x; i < G; i += 32) t += __ldcg(part + (size_t)j * kMaxBlocksPerSystem + i);
      tot[j] = warp_sum(t);
    }
  }
  if (threadIdx.x == 0) *ticket = 0u;
}

// Row range [e0, e1) of row i, or an empty range (and the bad-CSR flag) if row_ptr is out of bounds.
template <typename I>
__device__ __forceinline__ void row_range(const I *rp, int64_t i, int64_t nnz, int64_t &e0, int64_t &e1,
                                          uint32_t *bad) {
  e0 = (int64_t)rp[i];
  e1 = (int64_t)rp[i + 1];
  if (e0 < 0 || e1 < e0 || e1 > nnz) {
    if (bad) atomicOr(bad, 1u);
    e0 = e1 = 0;
  }
}

// True when column c is inside [0, n); otherwise raises the bad-CSR flag.
__device__ __forceinline__ bool col_ok(int32_t c, int32_t n, uint32_t *bad) {
  const bool ok = (uint32_t)c < (uint32_t)n;
  if (!ok && bad) atomicOr(bad, 1u);
  return ok;
}

__device__ __forceinline__ void count_kernel(Glob *g) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicAdd(&g->kernels, 1ull);
}

}  // namespace sla
