// Streaming loop over the stored entries of a CSR pattern, for the gradients that live on it.
//
// Both gradients of the method are one value per stored entry e = (i, j), in CSR order:
//   linear systems (Methodology 2):      grad_values[e] = -lambda_i * x_j
//   eigenvalue problems (Methodology 2): grad_values[e] = sum_s w_s v_s[i] v_s[j]
// ("torch-sla" technical summary).  Each is a product of a per-row factor and a gathered
// per-column value, so the work is one pass over col_idx (read) and grad_values (written),
// plus the row pointers and two vectors.
//
// Layout of the pass.  A block takes a tile of kPatRows consecutive rows: it stages their row
// pointers and row factors in shared memory (loaded one tile ahead into registers, coalesced, so
// their latency hides behind the previous tile), then walks the tile's entries in
// chunks of at most kPatChunk.  For a chunk, each row's thread writes the row's index into a
// per-entry table in shared memory; then every thread takes consecutive entries, kPatUnroll at a
// time (their col_idx loads, then their gathers, in flight together): coalesced col_idx loads and
// grad_values stores, the row factor from shared memory, the column value gathered from L2.
// Rows longer than a chunk are split across chunks; empty rows cost nothing.
//
// Malformed row pointers never cause an out-of-bounds access: the tile's entry range is clamped
// into [0, nnz], each row's range into the chunk, and a table slot no row wrote is clamped into
// the tile.  Such entries then get an unspecified (finite-input) value; columns out of [0, n)
// give 0.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sla {

#ifndef SLA_PAT_UNROLL
#define SLA_PAT_UNROLL 6
#endif
#ifndef SLA_PAT_MIN_BLOCKS
#define SLA_PAT_MIN_BLOCKS 5
#endif
constexpr int kPatBlock = 256;    // threads per block
constexpr int kPatRows = 256;     // rows per tile (small tiles: many per SM, a short tail wave)
constexpr int kPatChunk = 4096;   // entries per chunk (row-index table of 16-bit slots)
constexpr int kPatUnroll = SLA_PAT_UNROLL;  // entries per thread in flight
// resident blocks per SM the kernels are compiled for: the register budget this leaves (51 a thread)
// holds kPatUnroll entries in flight without spilling; with no minimum the compiler caps the
// kernels at 32 registers and spills
constexpr int kPatMinBlocks = SLA_PAT_MIN_BLOCKS;
static_assert(kPatRows <= 65536, "row index within a tile must fit 16 bits");

// Shared memory of one block: row pointers of the tile, row factors, the chunk's row-index table.
template <typename T>
struct PatSmem {
  int64_t rp[kPatRows + 1];
  T a[kPatRows];
  uint16_t rid[kPatChunk];
};

// rowload(i): the raw per-row input of global row i (a load, issued one tile ahead: its latency
// is hidden behind the current tile); rowprep(raw) -> T: the row's factor.  colload(c): the
// per-column value gathered for column c, called only for c in [0, n); the kUnroll gathers of a
// thread are issued together, before any entry is written.  entfn(e, i, a_i, c, v_c): writes
// entry e of row i, column c (v_c = 0 when c is out of [0, n)).  Tiles are taken round-robin by
// the blocks of the x dimension of the grid; each thread stages one row of a tile.
template <typename T, typename I, typename RowLoad, typename RowPrep, typename ColLoad, typename EntryFn>
__device__ __forceinline__ void pattern_pass(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                             const int32_t *__restrict__ ci, PatSmem<T> &sm, RowLoad rowload,
                                             RowPrep rowprep, ColLoad colload, EntryFn entfn) {
  static_assert(kPatRows == kPatBlock, "one row of a tile per thread");
  using R = decltype(rowload(int64_t(0)));
  using CV = decltype(colload(int32_t(0)));
  const int tid = threadIdx.x;
  const int64_t ntiles = (n + kPatRows - 1) / kPatRows;
  // this thread's row of the next tile (start pointer, raw input) and, in thread 0, the tile's end
  // (plain variables, not captured by a lambda, so that they stay in registers)
  int64_t nx_rp = 0, nx_end = 0;
  R nx_raw = R(0);
  if ((int64_t)blockIdx.x < ntiles) {
    const int64_t r0 = (int64_t)blockIdx.x * kPatRows;
    const int rows = (int)((n - r0) < kPatRows ? (n - r0) : kPatRows);
    if (tid < rows) {
      nx_rp = (int64_t)rp[r0 + tid];
      nx_raw = rowload(r0 + tid);
    }
    if (tid == 0) nx_end = (int64_t)rp[r0 + rows];
  }
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = t * kPatRows;
    const int rows = (int)((n - r0) < kPatRows ? (n - r0) : kPatRows);
    if (tid < rows) {
      sm.rp[tid] = nx_rp;
      sm.a[tid] = rowprep(nx_raw);
    }
    if (tid == 0) sm.rp[rows] = nx_end;
    __syncthreads();
    if (t + gridDim.x < ntiles) {  // the next tile's rows: in flight while this tile's entries run
      const int64_t r1 = (t + gridDim.x) * kPatRows;
      const int rows1 = (int)((n - r1) < kPatRows ? (n - r1) : kPatRows);
      if (tid < rows1) {
        nx_rp = (int64_t)rp[r1 + tid];
        nx_raw = rowload(r1 + tid);
      }
      if (tid == 0) nx_end = (int64_t)rp[r1 + rows1];
    }
    int64_t eb = sm.rp[0], ee = sm.rp[rows];
    if (eb < 0) eb = 0;
    if (ee > nnz) ee = nnz;
    for (int64_t c0 = eb; c0 < ee; c0 += kPatChunk) {
      const int64_t c1 = (ee - c0) < kPatChunk ? ee : c0 + kPatChunk;
      for (int j = tid; j < rows; j += kPatBlock) {
        const int64_t a = sm.rp[j] > c0 ? sm.rp[j] : c0;
        const int64_t b = sm.rp[j + 1] < c1 ? sm.rp[j + 1] : c1;
        for (int64_t e = a; e < b; ++e) sm.rid[e - c0] = (uint16_t)j;
      }
      __syncthreads();
      for (int64_t e0 = c0 + tid; e0 < c1; e0 += (int64_t)kPatUnroll * kPatBlock) {
        int32_t c[kPatUnroll];
#pragma unroll
        for (int u = 0; u < kPatUnroll; ++u) {
          const int64_t e = e0 + (int64_t)u * kPatBlock;
          c[u] = e < c1 ? __ldcs(ci + e) : -1;
        }
        CV v[kPatUnroll];
#pragma unroll
        for (int u = 0; u < kPatUnroll; ++u) v[u] = (uint32_t)c[u] < (uint32_t)n ? colload(c[u]) : CV(0);
#pragma unroll
        for (int u = 0; u < kPatUnroll; ++u) {
          const int64_t e = e0 + (int64_t)u * kPatBlock;
          if (e < c1) {
            int j = sm.rid[e - c0];
            if (j >= rows) j = rows - 1;
            entfn(e, r0 + j, sm.a[j], c[u], v[u]);
          }
        }
      }
      __syncthreads();
    }
    // every thread has read this tile's staged rows (also when it has no entries) before the next
    // tile overwrites them
    __syncthreads();
  }
}

}  // namespace sla
