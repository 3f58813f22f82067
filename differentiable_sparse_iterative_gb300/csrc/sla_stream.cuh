// The streaming CG kernels of the GRAPH and HOST loops (the host side is in sla_cg.cu).
//
// Method: "torch-sla" technical summary, Methodology 1-2 and Significance (Hestenes-Stiefel CG,
// optional Jacobi preconditioning, the adjoint solve by the same iteration).  Per iteration two
// fused kernels, cg_spmv_step (p update, delayed x update, q = A p, p.q) and cg_update_step
// (r update, r.r and r.z, beta and the stopping test), each ending in a deterministic last-block
// reduction; cg_init, cg_setup and cg_finish around the loop; cg_loop_control ends the graph's
// WHILE loop.  An opt-in TMA-staged variant of the SpMV step computes the same rows.
#pragma once

#include <cuda_runtime.h>

#include "sla_common.cuh"
#include "sla_tma.cuh"

namespace sla {

// ------------------------------------------------------------------------ kernels

// Launch shape of the two streaming kernels (compile-time; measured on GB300).
#ifndef SLA_SPMV_MIN_BLOCKS
#define SLA_SPMV_MIN_BLOCKS 8  // resident blocks per SM the SpMV step is compiled for (a full SM)
#endif
#ifndef SLA_SPMV_RPT
#define SLA_SPMV_RPT 2  // rows per thread per tile of the SpMV step
#endif
#ifndef SLA_UPD_ROWS
#define SLA_UPD_ROWS 8  // rows per thread whose loads the update step issues together
#endif
#ifndef SLA_UPD_MIN_BLOCKS
#define SLA_UPD_MIN_BLOCKS 4
#endif
#ifndef SLA_UPD_MIN_BLOCKS_JAC64
#define SLA_UPD_MIN_BLOCKS_JAC64 3  // fp64 with Jacobi: three loaded vectors per row need more registers
#endif

template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) cg_init(Prob<V, I> P) {
  // zero the control blocks; every system starts active
  for (int s = threadIdx.x; s < P.batch; s += kBlock) {
    Ctl c;
    memset(&c, 0, sizeof(c));
    P.ctl[s] = c;
  }
  if (threadIdx.x == 0) {
    P.glob->active = (uint32_t)P.batch;
    P.glob->bodies = 0;
    P.glob->kernels = 1ull;
    P.glob->safety_stop = 0;
    P.glob->bad_csr = 0;
  }
}

// Setup: x = x0 (or 0), r = b - A x0 (or b), Jacobi 1/A_ii, ||b||, r.r, r.z; then the
// stopping decisions of iteration 0.
template <typename V, typename I, bool JAC>
__global__ void __launch_bounds__(kBlock) cg_setup(Prob<V, I> P) {
  count_kernel(P.glob);
  const int s = blockIdx.y, bx = blockIdx.x;
  const int64_t vo = (int64_t)s * P.n;
  const V *val = P.val + s * P.val_stride;
  const V *b = P.b + vo;
  V *x = P.x + vo;
  V *r = P.r + vo;
  V *dinv = JAC ? P.dinv + vo : nullptr;
  const V *x0 = P.x0 ? P.x0 + vo : nullptr;
  int64_t c0, c1;
  chunk_of(P.n, P.G, bx, c0, c1);
  double acc[5] = {0.0, 0.0, 0.0, 0.0, 0.0};  // b.b, r.r, r.z, #non-finite diag, #diag <= 0
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kBlock) {
    const V bi = b[i];
    V ri = bi;
    int64_t e0, e1;
    row_range(P.rp, i, P.nnz, e0, e1, &P.glob->bad_csr);
    if (x0) {
      V s_ = V(0);
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = P.ci[e];
        if (col_ok(c, P.n, &P.glob->bad_csr)) s_ = fmav<V>(val[e], x0[c], s_);
      }
      ri = bi - s_;
      x[i] = x0[i];
    } else {
      x[i] = V(0);
    }
    r[i] = ri;
    acc[0] = fma((double)bi, (double)bi, acc[0]);
    acc[1] = fma((double)ri, (double)ri, acc[1]);
    if (JAC) {
      V d = V(0);
      for (int64_t e = e0; e < e1; ++e)
        if (P.ci[e] == (int32_t)i) d = val[e];
      if (!isfinite((double)d)) acc[3] += 1.0;
      else if (!(d > V(0))) acc[4] += 1.0;
      const V di = V(1) / d;
      dinv[i] = di;
      const V zi = di * ri;
      P.z[vo + i] = zi;
      acc[2] = fma((double)ri, (double)zi, acc[2]);
    }
  }
  block_sum<5>(acc);
  double *part = P.partials + (size_t)s * kRedSlots * kMaxBlocksPerSystem;
  Ctl *C = P.ctl + s;
  if (!publish_last<5>(acc, part, &C->ticket, P.G, bx)) return;
  double tot[5];
  reduce_partials<5>(part, P.G, &C->ticket, tot);
  if (threadIdx.x != 0) return;
  const double nb = sqrt(tot[0]);
  double *hist = P.history ? P.history + (size_t)s * (size_t)(P.maxit + 1) : nullptr;
  C->nb = nb;
  C->k = 0;
  int done = 1;
  if (!isfinite(nb)) {
    C->status = SLA_NONFINITE;
  } else if (nb == 0.0) {
    C->status = SLA_OK;
    C->pending = 2;
    C->rel_res = 0.0;
    if (hist) hist[0] = 0.0;
  } else if (JAC && tot[3] > 0.0) {
    C->status = SLA_NONFINITE;
  } else if (JAC && tot[4] > 0.0) {
    C->status = SLA_BREAKDOWN;
  } else {
    const double rr = tot[1];
    C->rel_res = sqrt(rr) / nb;
    if (hist) hist[0] = C->rel_res;
    if (!isfinite(rr)) {
      C->status = SLA_NONFINITE;
    } else if (sqrt(rr) <= P.rtol * nb) {
      C->status = SLA_OK;
    } else if (P.maxit == 0) {
      C->status = SLA_NOT_CONVERGED;
    } else {
      C->rho = JAC ? tot[2] : rr;
      C->status = SLA_NOT_CONVERGED;
      done = 0;
    }
  }
  if (done) {
    C->done = 1;
    atomicSub(&P.glob->active, 1u);
  }
}

// z_c = M^{-1} r_c and p_k[c] = z_c + beta p_{k-1}[c]: the same expression for rows of the tile
// (kept in shared memory) and for neighbours recomputed from global memory.
template <typename V>
__device__ __forceinline__ V p_of(const V *__restrict__ zs, const V *__restrict__ po, int64_t c, bool first, V beta) {
  const V zc = zs[c];
  return first ? zc : fmav<V>(beta, po[c], zc);
}

template <typename V, typename I, bool JAC, int RPT>
__global__ void __launch_bounds__(kBlock, SLA_SPMV_MIN_BLOCKS) cg_spmv_step(Prob<V, I> P, int par) {
  count_kernel(P.glob);
  const int s = blockIdx.y, bx = blockIdx.x;
  Ctl *C = P.ctl + s;
  if (C->done) return;
  const int64_t k = C->k;
  const bool first = (k == 0);
  const V beta = (V)C->beta;
  const V alpha_prev = (V)C->alpha;
  const int64_t vo = (int64_t)s * P.n;
  const V *__restrict__ val = P.val + s * P.val_stride;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  // z = M^{-1} r (r itself without a preconditioner)
  const V *__restrict__ zs = JAC ? P.z + vo : P.r + vo;
  const V *__restrict__ po = P.p[par ^ 1] + vo;
  V *__restrict__ pn = P.p[par] + vo;
  V *__restrict__ q = P.q + vo;
  V *__restrict__ x = P.x + vo;
  __shared__ V sp[kBlock * RPT];

  // Band sweep: tile t (T consecutive rows) belongs to block t mod G, so the grid walks the
  // vector as one band of G tiles.  The off-tile columns of a banded matrix (a grid stencil's
  // rows i +- m) then fall inside the band just read by other blocks and hit in L2, where
  // contiguous per-block chunks would re-read them from DRAM.  T is capped so that every block
  // has a tile when n is small.
  const int64_t per_block = ((int64_t)P.n + P.G - 1) / P.G;  // 64-bit: n may be close to 2^31
  const int64_t T = per_block < (int64_t)kBlock * RPT ? per_block : (int64_t)kBlock * RPT;
  const int64_t ntiles = (P.n + T - 1) / T;
  double pq = 0.0;
  for (int64_t t = bx; t < ntiles; t += P.G) {
    const int64_t s0 = t * T;
    const int len = (int)(P.n - s0 < T ? P.n - s0 : T);
    // loads of the tile's rows first (vectors and row pointers), then p_k, the delayed x update
    V zv[RPT], pov[RPT], xv[RPT];
    I rpa[RPT], rpb[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      const bool in = li < len;
      const int64_t i = s0 + li;
      zv[j] = in ? zs[i] : V(0);
      pov[j] = (in && !first) ? po[i] : V(0);
      xv[j] = (in && !first) ? x[i] : V(0);
      rpa[j] = in ? rp[i] : I(0);
      rpb[j] = in ? rp[i + 1] : I(0);
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const int64_t i = s0 + li;
        V pv = zv[j];
        if (!first) {
          pv = fmav<V>(beta, pov[j], zv[j]);
          x[i] = fmav<V>(alpha_prev, pov[j], xv[j]);
        }
        sp[li] = pv;
        pn[i] = pv;
      }
    }
    __syncthreads();
    V part = V(0);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const int64_t i = s0 + li;
        int64_t e0 = (int64_t)rpa[j], e1 = (int64_t)rpb[j];
        if (e0 < 0 || e1 < e0 || e1 > P.nnz) {
          atomicOr(&P.glob->bad_csr, 1u);
          e0 = e1 = 0;
        }
        V acc = V(0);
        for (int64_t e = e0; e < e1; ++e) {
          const int32_t c = ci[e];
          const V v = val[e];
          const uint32_t off = (uint32_t)((int64_t)c - s0);
          V pc;
          if (off < (uint32_t)len) pc = sp[off];
          else pc = col_ok(c, P.n, &P.glob->bad_csr) ? p_of<V>(zs, po, c, first, beta) : V(0);
          acc = fmav<V>(v, pc, acc);
        }
        q[i] = acc;
        part = fmav<V>(sp[li], acc, part);
      }
    }
    pq += (double)part;
    __syncthreads();
  }
  double v1[1] = {pq};
  block_sum<1>(v1);
  double *pp = P.partials + (size_t)s * kRedSlots * kMaxBlocksPerSystem;
  if (!publish_last<1>(v1, pp, &C->ticket, P.G, bx)) return;
  double tot[1];
  reduce_partials<1>(pp, P.G, &C->ticket, tot);
  if (threadIdx.x != 0) return;
  const double pqt = tot[0];
  int stop = 0;
  if (!isfinite(pqt)) {
    C->status = SLA_NONFINITE;
    stop = 1;
  } else if (!(pqt > 0.0)) {
    C->status = SLA_BREAKDOWN;
    stop = 1;
  } else {
    C->alpha = C->rho / pqt;
  }
  if (stop) {
    C->done = 1;
    C->pending = 0;
    atomicSub(&P.glob->active, 1u);
  }
}

// ---- TMA-staged SpMV step (same arithmetic as cg_spmv_step, same results bit for bit)
//
// The block walks its chunk in tiles of kTmaRows rows.  Thread 0 streams each tile's CSR
// entries (col_idx, values) and row vectors (z, p_{k-1}, x) into a shared-memory stage with
// 1-D bulk copies, two stages deep, so the copy of tile t+1 overlaps the arithmetic of tile t and
// the matrix stream never waits on per-thread loads.  Bulk copies need 16-byte alignment: each
// array's aligned interior is copied, the ragged ends (a few entries) are read from global
// memory directly, and a tile with more than kTmaCap entries reads its CSR entries from global
// memory.  A stage wait that exceeds its bound also falls back to global memory and raises the
// timeout flag, so results never depend on a copy completing.
constexpr int kTmaBlock = 512;         // threads per block of the TMA-staged step
constexpr int kTmaRows = kTmaBlock;    // rows per tile, one per thread
constexpr int kTmaCap = 6 * kTmaRows;  // CSR entries a stage holds
constexpr int kTmaRemote = 4;          // off-tile columns per row whose p is gathered ahead
constexpr long long kTmaWaitLimit = 1ll << 22;

template <typename V>
struct __align__(16) TmaStage {
  static constexpr int kEv = 16 / (int)sizeof(V);  // elements per 16 bytes
  alignas(16) int32_t ci[kTmaCap + 8];
  alignas(16) V val[kTmaCap + 2 * kEv];
  alignas(16) V zv[kTmaRows + 2 * kEv];
  alignas(16) V pov[kTmaRows + 2 * kEv];
  alignas(16) V xv[kTmaRows + 2 * kEv];
};

// What a stage holds: aligned interiors [a, b) of the entry range and of the row range, with the
// index of element 0 of each staged array (base).  Written by thread 0 before the copies.
struct TmaPlan {
  int64_t cbase, ca, cb;   // col_idx entries
  int64_t vbase, va, vb;   // values entries
  int64_t rbase, ra, rb;   // rows (z, p_{k-1}, x)
  int fallback;            // 1: CSR entries not staged for this tile
};

__device__ __forceinline__ int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
__device__ __forceinline__ int64_t round_dn(int64_t v, int64_t m) { return v / m * m; }

template <typename V>
__host__ __device__ constexpr size_t tma_smem_bytes() {
  return 2 * sizeof(TmaStage<V>) + (size_t)kTmaRows * sizeof(V);
}

// Thread 0: plan and issue the copies of one tile into one stage.
template <typename V>
__device__ __forceinline__ void tma_issue(TmaStage<V> &st, TmaPlan &pl, uint64_t *bar, const int32_t *ci,
                                          const V *val, const V *zs, const V *po, const V *x, int64_t s0, int len,
                                          int64_t e_lo, int64_t e_hi, int64_t nnz, bool first) {
  constexpr int kEv = TmaStage<V>::kEv;
  uint32_t bytes = 0;
  // never copy outside [0, nnz): a malformed row_ptr makes the tile read global memory, where
  // the per-row checks skip out-of-range entries
  pl.fallback = (e_hi - e_lo > kTmaCap || e_lo < 0 || e_hi < e_lo || e_hi > nnz) ? 1 : 0;
  if (pl.fallback) e_lo = e_hi = 0;
  pl.cbase = round_dn(e_lo, 4);
  pl.ca = round_up(e_lo, 4);
  pl.cb = round_dn(e_hi, 4);
  pl.vbase = round_dn(e_lo, kEv);
  pl.va = round_up(e_lo, kEv);
  pl.vb = round_dn(e_hi, kEv);
  if (pl.fallback || pl.cb < pl.ca) pl.cb = pl.ca;
  if (pl.fallback || pl.vb < pl.va) pl.vb = pl.va;
  pl.rbase = round_dn(s0, kEv);
  pl.ra = round_up(s0, kEv);
  pl.rb = round_dn(s0 + len, kEv);
  if (pl.rb < pl.ra) pl.rb = pl.ra;
  const uint32_t cbytes = (uint32_t)((pl.cb - pl.ca) * 4);
  const uint32_t vbytes = (uint32_t)((pl.vb - pl.va) * (int64_t)sizeof(V));
  const uint32_t rbytes = (uint32_t)((pl.rb - pl.ra) * (int64_t)sizeof(V));
  bytes = cbytes + vbytes + rbytes * (first ? 1u : 3u);
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(bar, bytes);
  if (cbytes) bulk_g2s(st.ci + (pl.ca - pl.cbase), ci + pl.ca, cbytes, bar);
  if (vbytes) bulk_g2s(st.val + (pl.va - pl.vbase), val + pl.va, vbytes, bar);
  if (rbytes) {
    bulk_g2s(st.zv + (pl.ra - pl.rbase), zs + pl.ra, rbytes, bar);
    if (!first) {
      bulk_g2s(st.pov + (pl.ra - pl.rbase), po + pl.ra, rbytes, bar);
      bulk_g2s(st.xv + (pl.ra - pl.rbase), x + pl.ra, rbytes, bar);
    }
  }
}

template <typename V, typename I, bool JAC>
__global__ void __launch_bounds__(kTmaBlock, 2) cg_spmv_step_tma(Prob<V, I> P, int par) {
  count_kernel(P.glob);
  const int s = blockIdx.y, bx = blockIdx.x;
  Ctl *C = P.ctl + s;
  if (C->done) return;
  extern __shared__ __align__(16) unsigned char tma_smem[];
  TmaStage<V> *stage = reinterpret_cast<TmaStage<V> *>(tma_smem);
  V *sp = reinterpret_cast<V *>(tma_smem + 2 * sizeof(TmaStage<V>));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ TmaPlan plan[2];

  const int64_t k = C->k;
  const bool first = (k == 0);
  const V beta = (V)C->beta;
  const V alpha_prev = (V)C->alpha;
  const int64_t vo = (int64_t)s * P.n;
  const V *__restrict__ val = P.val + s * P.val_stride;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *__restrict__ zs = JAC ? P.z + vo : P.r + vo;
  const V *__restrict__ po = P.p[par ^ 1] + vo;
  V *__restrict__ pn = P.p[par] + vo;
  V *__restrict__ q = P.q + vo;
  V *__restrict__ x = P.x + vo;

  int64_t c0, c1;
  chunk_of(P.n, P.G, bx, c0, c1);
  const int ntiles = (int)((c1 - c0 + kTmaRows - 1) / kTmaRows);
  auto tile_s0 = [&](int t) { return c0 + (int64_t)t * kTmaRows; };
  auto tile_len = [&](int t) { return (int)min((int64_t)kTmaRows, c1 - tile_s0(t)); };

  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_proxy_async_smem();
    for (int t = 0; t < 2 && t < ntiles; ++t) {
      const int64_t a = tile_s0(t);
      const int l = tile_len(t);
      tma_issue<V>(stage[t], plan[t], &bar[t], ci, val, zs, po, x, a, l, (int64_t)rp[a], (int64_t)rp[a + l], P.nnz,
                   first);
    }
  }
  __syncthreads();

  bool late = false;  // a stage wait ran out: read global memory for that tile
  double pq = 0.0;
  const int li = threadIdx.x;  // the thread's row within each tile
  for (int t = 0; t < ntiles; ++t) {
    const int sidx = t & 1;
    const uint32_t parity = (uint32_t)((t >> 1) & 1);
    const int64_t s0 = tile_s0(t);
    const int len = tile_len(t);
    const bool mine = li < len;
    const int64_t i = s0 + li;
    // bounds of tile t+2 for the producer, and this row's pointers, before the wait
    int64_t nlo = 0, nhi = 0;
    if (threadIdx.x == 0 && t + 2 < ntiles) {
      const int64_t a = tile_s0(t + 2);
      nlo = (int64_t)rp[a];
      nhi = (int64_t)rp[a + tile_len(t + 2)];
    }
    int64_t e0 = mine ? (int64_t)rp[i] : 0, e1 = mine ? (int64_t)rp[i + 1] : 0;
    if (e0 < 0 || e1 < e0 || e1 > P.nnz) {
      atomicOr(&P.glob->bad_csr, 1u);
      e0 = e1 = 0;
    }
    const bool ok = mbar_wait_bounded(&bar[sidx], parity, kTmaWaitLimit);
    if (!ok) {
      late = true;
      atomicOr(&P.glob->timeout, 1u);
    }
    const TmaStage<V> &st = stage[sidx];
    const TmaPlan pl = plan[sidx];
    const bool staged_csr = ok && !pl.fallback;
    // gather ahead: z and p_{k-1} at this row's first kTmaRemote off-tile columns
    V rz[kTmaRemote], rpo[kTmaRemote];
    int nrem = 0;
    for (int64_t e = e0; e < e1 && nrem < kTmaRemote; ++e) {
      const int32_t c = (staged_csr && e >= pl.ca && e < pl.cb) ? st.ci[e - pl.cbase] : ci[e];
      if ((uint32_t)((int64_t)c - s0) >= (uint32_t)len && (uint32_t)c < (uint32_t)P.n) {
#pragma unroll
        for (int u = 0; u < kTmaRemote; ++u)
          if (u == nrem) {
            rz[u] = zs[c];
            rpo[u] = first ? V(0) : po[c];
          }
        ++nrem;
      }
    }
    // p_k for the row and the delayed x update
    if (mine) {
      const bool in = ok && i >= pl.ra && i < pl.rb;
      const V zi = in ? st.zv[i - pl.rbase] : zs[i];
      V pv = zi;
      if (!first) {
        const V pold = in ? st.pov[i - pl.rbase] : po[i];
        const V xo = in ? st.xv[i - pl.rbase] : x[i];
        pv = fmav<V>(beta, pold, zi);
        x[i] = fmav<V>(alpha_prev, pold, xo);
      }
      sp[li] = pv;
      pn[i] = pv;
    }
    __syncthreads();
    V part = V(0);
    if (mine) {
      V acc = V(0);
      int used = 0;
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = (staged_csr && e >= pl.ca && e < pl.cb) ? st.ci[e - pl.cbase] : ci[e];
        const V v = (staged_csr && e >= pl.va && e < pl.vb) ? st.val[e - pl.vbase] : val[e];
        const uint32_t off = (uint32_t)((int64_t)c - s0);
        V pc;
        if (off < (uint32_t)len) {
          pc = sp[off];
        } else if (!col_ok(c, P.n, &P.glob->bad_csr)) {
          pc = V(0);
        } else if (used < nrem) {
          V zc = rz[0], pc0 = rpo[0];
#pragma unroll
          for (int u = 1; u < kTmaRemote; ++u)
            if (u == used) {
              zc = rz[u];
              pc0 = rpo[u];
            }
          pc = first ? zc : fmav<V>(beta, pc0, zc);
          ++used;
        } else {
          pc = p_of<V>(zs, po, c, first, beta);
        }
        acc = fmav<V>(v, pc, acc);
      }
      q[i] = acc;
      part = fmav<V>(sp[li], acc, part);
    }
    pq += (double)part;
    __syncthreads();  // the stage and sp are free again
    if (threadIdx.x == 0 && t + 2 < ntiles) {
      if (late) {
        // the previous copy into this stage may still be in flight: let it land first
        mbar_wait_bounded(&bar[sidx], parity, kTmaWaitLimit);
      }
      tma_issue<V>(stage[sidx], plan[sidx], &bar[sidx], ci, val, zs, po, x, tile_s0(t + 2), tile_len(t + 2), nlo,
                   nhi, P.nnz, first);
    }
  }
  if (late && threadIdx.x == 0) {
    // no copy may outlive the block
    for (int t = ntiles - 2; t < ntiles; ++t)
      if (t >= 0) mbar_wait_bounded(&bar[t & 1], (uint32_t)((t >> 1) & 1), kTmaWaitLimit);
  }
  double v1[1] = {pq};
  block_sum_n<1, kTmaBlock>(v1);
  double *pp = P.partials + (size_t)s * kRedSlots * kMaxBlocksPerSystem;
  if (!publish_last<1>(v1, pp, &C->ticket, P.G, bx)) return;
  double tot[1];
  reduce_partials<1>(pp, P.G, &C->ticket, tot);
  if (threadIdx.x != 0) return;
  const double pqt = tot[0];
  int stop = 0;
  if (!isfinite(pqt)) {
    C->status = SLA_NONFINITE;
    stop = 1;
  } else if (!(pqt > 0.0)) {
    C->status = SLA_BREAKDOWN;
    stop = 1;
  } else {
    C->alpha = C->rho / pqt;
  }
  if (stop) {
    C->done = 1;
    C->pending = 0;
    atomicSub(&P.glob->active, 1u);
  }
}

template <typename V, typename I, bool JAC>
__global__ void __launch_bounds__(kBlock, (JAC && sizeof(V) == 8) ? SLA_UPD_MIN_BLOCKS_JAC64 : SLA_UPD_MIN_BLOCKS)
    cg_update_step(Prob<V, I> P, int par) {
  count_kernel(P.glob);
  const int s = blockIdx.y, bx = blockIdx.x;
  Ctl *C = P.ctl + s;
  if (C->done) return;
  const V alpha = (V)C->alpha;
  const int64_t vo = (int64_t)s * P.n;
  V *__restrict__ r = P.r + vo;
  const V *__restrict__ q = P.q + vo;
  const V *__restrict__ dinv = JAC ? P.dinv + vo : nullptr;
  V *__restrict__ z = JAC ? P.z + vo : nullptr;
  // groups of kUpd rows per thread: all loads of a group first, then the arithmetic.  When every
  // block has many groups, chunks are whole groups except the last block's (no block ends in a
  // partly empty group); with few groups per block that rounding would unbalance the blocks.
  constexpr int kUpd = SLA_UPD_ROWS;
  constexpr int64_t kGroupRows = (int64_t)kUpd * kBlock;
  int64_t c0, c1;
  if ((int64_t)P.n >= 16 * kGroupRows * (int64_t)P.G) chunk_aligned(P.n, P.G, bx, kGroupRows, c0, c1);
  else chunk_of(P.n, P.G, bx, c0, c1);
  double acc[2] = {0.0, 0.0};
  for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kUpd * kBlock) {
    V qv[kUpd], rv[kUpd], dv[kUpd];
#pragma unroll
    for (int u = 0; u < kUpd; ++u) {
      const int64_t i = g0 + (int64_t)u * kBlock;
      const bool in = i < c1;
      qv[u] = in ? q[i] : V(0);
      rv[u] = in ? r[i] : V(0);
      if (JAC) dv[u] = in ? dinv[i] : V(0);
    }
    // fp64 data accumulates straight into the fp64 sums; fp32 data per group in fp32 first
    V rr = V(0), rz = V(0);
    if constexpr (sizeof(V) == 8) {
      rr = acc[0];
      rz = acc[1];
    }
#pragma unroll
    for (int u = 0; u < kUpd; ++u) {
      const int64_t i = g0 + (int64_t)u * kBlock;
      if (i < c1) {
        const V ri = fmav<V>(-alpha, qv[u], rv[u]);
        r[i] = ri;
        rr = fmav<V>(ri, ri, rr);
        if (JAC) {
          const V zi = dv[u] * ri;
          z[i] = zi;
          rz = fmav<V>(ri, zi, rz);
        }
      }
    }
    if constexpr (sizeof(V) == 8) {
      acc[0] = rr;
      acc[1] = rz;
    } else {
      acc[0] += (double)rr;
      if (JAC) acc[1] += (double)rz;
    }
  }
  block_sum<2>(acc);
  double *pp = P.partials + (size_t)s * kRedSlots * kMaxBlocksPerSystem;
  if (!publish_last<2>(acc, pp, &C->ticket, P.G, bx)) return;
  double tot[2];
  reduce_partials<2>(pp, P.G, &C->ticket, tot);
  if (threadIdx.x != 0) return;
  const double rrt = tot[0];
  const int64_t k1 = C->k + 1;
  C->k = k1;
  C->rel_res = sqrt(rrt) / C->nb;
  if (P.history) P.history[(size_t)s * (size_t)(P.maxit + 1) + (size_t)k1] = C->rel_res;
  C->last_parity = par;
  int stop = 1;
  if (!isfinite(rrt)) {
    C->status = SLA_NONFINITE;
  } else if (sqrt(rrt) <= P.rtol * C->nb) {
    C->status = SLA_OK;
  } else if (k1 >= P.maxit) {
    C->status = SLA_NOT_CONVERGED;
  } else {
    const double rho_new = JAC ? tot[1] : rrt;
    C->beta = rho_new / C->rho;
    C->rho = rho_new;
    stop = 0;
  }
  if (stop) {
    C->done = 1;
    C->pending = 1;  // x += alpha_k p_k still to apply
    atomicSub(&P.glob->active, 1u);
  }
}

// Ends the device-side loop once every system has stopped (or, as a guard that should never
// fire, after more bodies than maxit allows).
__global__ void cg_loop_control(Glob *g, cudaGraphConditionalHandle h, uint32_t max_bodies) {
  if (threadIdx.x == 0) {
    atomicAdd(&g->kernels, 1ull);
    const uint32_t bodies = ++g->bodies;
    const uint32_t active = *(volatile uint32_t *)&g->active;
    if (active == 0u || bodies >= max_bodies) {
      if (active != 0u) g->safety_stop = 1u;
      cudaGraphSetConditional(h, 0u);
    }
  }
}

template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) cg_finish(Prob<V, I> P) {
  count_kernel(P.glob);
  const int s = blockIdx.y, bx = blockIdx.x;
  const Ctl *C = P.ctl + s;
  const int pending = C->pending;
  if (pending == 0) return;
  const int64_t vo = (int64_t)s * P.n;
  V *x = P.x + vo;
  const V *p = P.p[C->last_parity] + vo;
  const V alpha = (V)C->alpha;
  int64_t c0, c1;
  chunk_of(P.n, P.G, bx, c0, c1);
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kBlock)
    x[i] = pending == 1 ? fmav<V>(alpha, p[i], x[i]) : V(0);
}

}  // namespace sla
