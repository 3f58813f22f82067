// BiCGStab solve of a general (non-symmetric) sparse system and its adjoint backward (libsla).
//
// Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers and Sparse
// Tensor Parallelism for PyTorch" (Chi, Wen), technical summary: Methodology 1 lists BiCGStab
// among the solvers behind .solve; Methodology 2 gives the adjoint of x = A^{-1} b for any A:
// A^T lambda = dL/dx, grad_b = lambda, grad_A = -lambda_i x_j on the sparsity pattern.  The
// iteration is the textbook one (H. A. van der Vorst, "Bi-CGSTAB", SIAM J. Sci. Stat. Comput. 13,
// 1992), unpreconditioned, with the shadow residual rhat = r_0:
//   rho = rhat.r; p = r (first) or r + beta (p - omega v), beta = (rho / rho_prev)(alpha / omega);
//   v = A p; alpha = rho / rhat.v; s = r - alpha v (stop with x += alpha p when ||s|| <= rtol ||b||);
//   t = A s; omega = t.s / t.t; x += alpha p + omega s; r = s - omega t; stop when
//   ||r|| <= rtol ||b||.  Zero rhat.v, t.t, omega or rho is a breakdown.
//
// GB300 design.  Two engines.  The default runs the whole solve in one cooperative kernel
// (bi_resident, described with it below).  The host loop, for profiling and for GPUs where the
// cooperative launch is refused, runs three kernels per iteration: bi_dir_apply forms the
// direction p and v = A p with rhat.v; bi_s_apply forms s = r - alpha v and t = A s with s.s, t.s
// and t.t; bi_update the x and r updates with rhat.r and r.r.  The two product kernels walk the rows in tiles dealt to the
// blocks round-robin (a band sweep: a stencil's off-tile neighbours were just read by the blocks
// beside it and hit in L2); a tile's own p (or s) stays in shared memory for the product, and a
// neighbour's is recomputed from r, p_prev and v_prev (or r and v) by the same expression, so
// the vector is never re-read after it is written.  p and v are double-buffered (the recomputation
// reads the previous iteration's).  Every thread issues the loads of all its rows before their
// arithmetic.  Dot products are summed in fp64 in a fixed order (a block sum per block, then the
// last block to arrive adds the block sums in index order) and every scalar decision is taken by
// that block on the device, so the host only enqueues `unroll` iterations at a time and reads the
// state between them; the kernels of a finished solve return at once.  The adjoint runs the same
// kernels on A's pattern with every value taken from its partner entry (j, i) when the pattern is
// structurally symmetric, and on an explicitly built A^T otherwise.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "sla_common.cuh"
#include "sla_grid.cuh"
#include "sla_host.h"

namespace sla {
namespace {

// Device state of one solve.
struct BiCtl {
  double nb, rho, alpha, omega, beta, ss, rel;
  int64_t k, maxit;
  double rtol;
  int32_t status, done;
  int32_t exit_s;   // this iteration's s passed the stopping test: x += alpha p, r = s
  int32_t zero_x;   // b = 0: x = 0 at the end
  uint32_t ticket;  // arrival counter of the last-block reductions
  uint32_t bad;     // a row range, a column index or (adjoint) a partner entry was missing
  uint32_t arrive;  // grid-barrier arrivals of the resident kernel
  uint32_t timeout; // a grid-barrier wait of the resident kernel expired
  uint32_t nopartner;  // (adjoint) an entry (i, j) has no stored (j, i): A^T is built explicitly
};

// Rows of block partial sums: the streaming kernels use rows 0-2; the resident kernel gives each
// phase its own rows (setup 0-1, rhat.v 2, s.s / t.s / t.t 3-5, rhat.r / r.r 6-7) so that a block
// already in the next phase never overwrites sums that another block is still reading.
constexpr int kBiSlots = 8;

// Rows of the explicit transpose's column-count scan handled by one block.
constexpr int64_t kTrChunk = 4096;

struct BiLayout {
  size_t ctl, part, r, rh, p[2], v[2], s, t, vt;
  size_t tp, tci, cnt, bsum;  // the adjoint's explicit A^T (patterns without partner entries)
  size_t total;
};

BiLayout bi_layout(int64_t n, int64_t nnz, size_t vsz) {
  BiLayout L;
  size_t off = 0;
  const size_t vec = align256(vsz * (size_t)n);
  L.ctl = off; off += align256(sizeof(BiCtl));
  L.part = off; off += align256(sizeof(double) * kBiSlots * (size_t)kMaxBlocksPerSystem);
  L.r = off; off += vec;
  L.rh = off; off += vec;
  L.p[0] = off; off += vec;
  L.p[1] = off; off += vec;
  L.v[0] = off; off += vec;
  L.v[1] = off; off += vec;
  L.s = off; off += vec;
  L.t = off; off += vec;
  L.vt = off; off += align256(vsz * (size_t)nnz);  // the adjoint's transposed values
  L.tp = off; off += align256(sizeof(int64_t) * ((size_t)n + 1));  // A^T row pointers (as A's type)
  L.tci = off; off += align256(sizeof(int32_t) * (size_t)nnz);     // A^T column indices
  L.cnt = off; off += align256(sizeof(int32_t) * (size_t)n);       // column counts, then cursors
  L.bsum = off; off += align256(sizeof(int64_t) * (size_t)((n + kTrChunk - 1) / kTrChunk + 1));
  L.total = off;
  return L;
}

// Rows per thread of a tile of the two product kernels, and of a load group of bi_update.
constexpr int kBiRPT = 2;
constexpr int kBiTile = kBlock * kBiRPT;
constexpr int kBiUpd = 4;
constexpr int kBiProdBlocks = 8;  // resident blocks per SM the product kernels are compiled for
constexpr int kBiUpdBlocks = 4;   // and bi_update (five vectors of kBiUpd rows in flight per thread)

int bi_sms() {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Blocks of the product kernels: the tiles of kBiTile rows shared out evenly over at most one full
// wave and no more blocks than the partial-sum slots hold.
int bi_grid(int64_t n) {
  int64_t cap = (int64_t)bi_sms() * kBiProdBlocks;
  if (cap > kMaxBlocksPerSystem) cap = kMaxBlocksPerSystem;
  const int64_t tiles = (n + kBiTile - 1) / kBiTile;
  if (tiles <= cap) return tiles < 1 ? 1 : (int)tiles;
  const int64_t per = (tiles + cap - 1) / cap;  // tiles per block
  return (int)((tiles + per - 1) / per);
}

// Blocks of bi_update: one full wave, fewer when n gives a block less than one group per thread.
int bi_upd_grid(int64_t n) {
  int64_t g = (n + (int64_t)kBlock * kBiUpd - 1) / ((int64_t)kBlock * kBiUpd);
  const int64_t cap = (int64_t)bi_sms() * kBiUpdBlocks;
  if (g > cap) g = cap;
  if (g > kMaxBlocksPerSystem) g = kMaxBlocksPerSystem;
  return g < 1 ? 1 : (int)g;
}

template <typename V, typename I>
struct BiProb {
  int64_t n, nnz;
  const I *rp;
  const int32_t *ci;
  const V *val;
  const V *b;
  const V *x0;
  V *x, *r, *rh, *p[2], *v[2], *s, *t;
  double *part;
  double *hist;
  BiCtl *C;
};

template <typename V, typename I>
__device__ __forceinline__ V row_times(const BiProb<V, I> &P, int64_t i, const V *y) {
  int64_t e0, e1;
  row_range(P.rp, i, P.nnz, e0, e1, &P.C->bad);
  V acc = V(0);
  for (int64_t e = e0; e < e1; ++e) {
    const int32_t c = P.ci[e];
    if (col_ok(c, (int32_t)P.n, &P.C->bad)) acc = fmav<V>(P.val[e], y[c], acc);
  }
  return acc;
}

#define BI_ROWS(i) for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < P.n; i += (int64_t)gridDim.x * kBlock)

// r = b - A x0 (r = b), x = x0 (0), rhat = r; ||b|| and r.r; the decisions before the first iteration.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) bi_setup(BiProb<V, I> P) {
  double acc[2] = {0.0, 0.0};
  BI_ROWS(i) {
    const V bi = P.b[i];
    V ri = bi;
    if (P.x0) ri = bi - row_times(P, i, P.x0);
    const V xi = P.x0 ? P.x0[i] : V(0);
    P.r[i] = ri;
    P.rh[i] = ri;
    acc[0] = fma((double)bi, (double)bi, acc[0]);
    acc[1] = fma((double)ri, (double)ri, acc[1]);
    P.x[i] = xi;  // x may be x0's own buffer: the same value, and the rows' products read x0 above
  }
  block_sum<2>(acc);
  if (!publish_last<2>(acc, P.part, &P.C->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[2];
  reduce_partials<2>(P.part, (int)gridDim.x, &P.C->ticket, tot);
  if (threadIdx.x != 0) return;
  BiCtl &C = *P.C;
  const double nb = sqrt(tot[0]), rr = tot[1];
  C.nb = nb;
  C.k = 0;
  C.alpha = C.omega = 1.0;
  C.beta = 0.0;
  C.rho = rr;  // rhat.r with rhat = r: the same sum
  C.exit_s = 0;
  C.zero_x = 0;
  C.status = SLA_NOT_CONVERGED;
  C.done = 0;
  if (!isfinite(nb)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (nb == 0.0) {
    C.rel = 0.0;
    if (P.hist) P.hist[0] = 0.0;
    C.zero_x = 1;
    C.status = SLA_OK;
    C.done = 1;
    return;
  }
  C.rel = sqrt(rr) / nb;
  if (P.hist) P.hist[0] = C.rel;
  if (!isfinite(rr)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (sqrt(rr) <= C.rtol * nb) { C.status = SLA_OK; C.done = 1; return; }
  if (C.maxit == 0) { C.done = 1; return; }
}

// Tile geometry of the product kernels: tile t (T consecutive rows) belongs to block t mod G; T is
// capped so that every block has a tile when n is small.
struct BiTiles {
  int64_t T, ntiles;
};

__device__ __forceinline__ BiTiles bi_tiles(int64_t n) {
  const int64_t G = gridDim.x;
  const int64_t per_block = (n + G - 1) / G;
  BiTiles tl;
  tl.T = per_block < (int64_t)kBiTile ? per_block : (int64_t)kBiTile;
  tl.ntiles = (n + tl.T - 1) / tl.T;
  return tl;
}

// p_c = r_c (first iteration) or r_c + beta (p_prev_c - omega v_prev_c): one expression for a
// tile's rows and for recomputed neighbours.
template <typename V>
__device__ __forceinline__ V p_at(V rc, V pc, V vc, bool first, V beta, V omega) {
  return first ? rc : fmav<V>(beta, fmav<V>(-omega, vc, pc), rc);
}

// The direction p and v = A p, rhat.v; alpha = rho / rhat.v.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock, kBiProdBlocks) bi_dir_apply(BiProb<V, I> P) {
  const BiCtl &Cr = *P.C;
  if (Cr.done) return;
  const int par = (int)(Cr.k & 1);
  const bool first = Cr.k == 0;
  const V beta = (V)Cr.beta, omega = (V)Cr.omega;
  const int64_t n = P.n;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *__restrict__ val = P.val;
  const V *__restrict__ r = P.r;
  const V *__restrict__ rh = P.rh;
  const V *__restrict__ po = P.p[par ^ 1];
  const V *__restrict__ vo = P.v[par ^ 1];
  V *__restrict__ pn = P.p[par];
  V *__restrict__ vn = P.v[par];
  __shared__ V sp[kBiTile];
  const BiTiles tl = bi_tiles(n);
  double acc = 0.0;
  for (int64_t tt = blockIdx.x; tt < tl.ntiles; tt += gridDim.x) {
    const int64_t s0 = tt * tl.T;
    const int len = (int)(n - s0 < tl.T ? n - s0 : tl.T);
    V rv[kBiRPT], pv[kBiRPT], vv[kBiRPT];
    I ra[kBiRPT], rb[kBiRPT];
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      const bool in = li < len;
      const int64_t i = s0 + li;
      rv[j] = in ? r[i] : V(0);
      pv[j] = (in && !first) ? po[i] : V(0);
      vv[j] = (in && !first) ? vo[i] : V(0);
      ra[j] = in ? rp[i] : I(0);
      rb[j] = in ? rp[i + 1] : I(0);
    }
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const V pi = p_at<V>(rv[j], pv[j], vv[j], first, beta, omega);
        sp[li] = pi;
        pn[s0 + li] = pi;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const int64_t i = s0 + li;
        int64_t e0 = (int64_t)ra[j], e1 = (int64_t)rb[j];
        if (e0 < 0 || e1 < e0 || e1 > P.nnz) {
          atomicOr(&P.C->bad, 1u);
          e0 = e1 = 0;
        }
        V a = V(0);
        for (int64_t e = e0; e < e1; ++e) {
          const int32_t c = ci[e];
          const V w = val[e];
          const uint32_t off = (uint32_t)((int64_t)c - s0);
          V pc;
          if (off < (uint32_t)len) pc = sp[off];
          else pc = col_ok(c, (int32_t)n, &P.C->bad) ? p_at<V>(r[c], first ? V(0) : po[c], first ? V(0) : vo[c],
                                                               first, beta, omega)
                                                     : V(0);
          a = fmav<V>(w, pc, a);
        }
        vn[i] = a;
        acc = fma((double)rh[i], (double)a, acc);
      }
    }
    __syncthreads();
  }
  double red[1] = {acc};
  block_sum<1>(red);
  if (!publish_last<1>(red, P.part, &P.C->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[1];
  reduce_partials<1>(P.part, (int)gridDim.x, &P.C->ticket, tot);
  if (threadIdx.x != 0) return;
  BiCtl &C = *P.C;
  const double rv = tot[0];
  if (!isfinite(rv)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (rv == 0.0) { C.status = SLA_BREAKDOWN; C.done = 1; return; }
  C.alpha = C.rho / rv;
}

// s = r - alpha v and t = A s; s.s, t.s and t.t.  The stopping test on ||s|| comes first (x += alpha p,
// r = s, and t unused), then omega = t.s / t.t.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock, kBiProdBlocks) bi_s_apply(BiProb<V, I> P) {
  const BiCtl &Cr = *P.C;
  if (Cr.done) return;
  const int par = (int)(Cr.k & 1);
  const V alpha = (V)Cr.alpha;
  const int64_t n = P.n;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *__restrict__ val = P.val;
  const V *__restrict__ r = P.r;
  const V *__restrict__ v = P.v[par];
  V *__restrict__ sg = P.s;
  V *__restrict__ tg = P.t;
  __shared__ V ss_[kBiTile];
  const BiTiles tl = bi_tiles(n);
  double acc[3] = {0.0, 0.0, 0.0};  // s.s, t.s, t.t
  for (int64_t tt = blockIdx.x; tt < tl.ntiles; tt += gridDim.x) {
    const int64_t s0 = tt * tl.T;
    const int len = (int)(n - s0 < tl.T ? n - s0 : tl.T);
    V rv[kBiRPT], vv[kBiRPT];
    I ra[kBiRPT], rb[kBiRPT];
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      const bool in = li < len;
      const int64_t i = s0 + li;
      rv[j] = in ? r[i] : V(0);
      vv[j] = in ? v[i] : V(0);
      ra[j] = in ? rp[i] : I(0);
      rb[j] = in ? rp[i + 1] : I(0);
    }
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const V si = fmav<V>(-alpha, vv[j], rv[j]);
        ss_[li] = si;
        sg[s0 + li] = si;
        acc[0] = fma((double)si, (double)si, acc[0]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kBiRPT; ++j) {
      const int li = j * kBlock + threadIdx.x;
      if (li < len) {
        const int64_t i = s0 + li;
        int64_t e0 = (int64_t)ra[j], e1 = (int64_t)rb[j];
        if (e0 < 0 || e1 < e0 || e1 > P.nnz) {
          atomicOr(&P.C->bad, 1u);
          e0 = e1 = 0;
        }
        V a = V(0);
        for (int64_t e = e0; e < e1; ++e) {
          const int32_t c = ci[e];
          const V w = val[e];
          const uint32_t off = (uint32_t)((int64_t)c - s0);
          V sc;
          if (off < (uint32_t)len) sc = ss_[off];
          else sc = col_ok(c, (int32_t)n, &P.C->bad) ? fmav<V>(-alpha, v[c], r[c]) : V(0);
          a = fmav<V>(w, sc, a);
        }
        tg[i] = a;
        const double sd = (double)ss_[li];
        acc[1] = fma((double)a, sd, acc[1]);
        acc[2] = fma((double)a, (double)a, acc[2]);
      }
    }
    __syncthreads();
  }
  block_sum<3>(acc);
  if (!publish_last<3>(acc, P.part, &P.C->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[3];
  reduce_partials<3>(P.part, (int)gridDim.x, &P.C->ticket, tot);
  if (threadIdx.x != 0) return;
  BiCtl &C = *P.C;
  C.ss = tot[0];
  if (!isfinite(C.ss)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  C.exit_s = sqrt(C.ss) <= C.rtol * C.nb ? 1 : 0;
  if (C.exit_s) return;
  if (!isfinite(tot[1]) || !isfinite(tot[2])) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (tot[2] == 0.0) { C.status = SLA_BREAKDOWN; C.done = 1; return; }
  C.omega = tot[1] / tot[2];
}

// x += alpha p + omega s, r = s - omega t (or x += alpha p, r = s after the early test); rhat.r,
// r.r; the stopping test and the next beta.  Each block takes a contiguous chunk of rows in
// groups of kBiUpd rows per thread, all loads of a group first.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock, kBiUpdBlocks) bi_update(BiProb<V, I> P) {
  const BiCtl &Cr = *P.C;
  if (Cr.done) return;
  const int par = (int)(Cr.k & 1);
  const bool ex = Cr.exit_s != 0;
  const V alpha = (V)Cr.alpha, omega = (V)Cr.omega;
  V *__restrict__ x = P.x;
  V *__restrict__ r = P.r;
  const V *__restrict__ p = P.p[par];
  const V *__restrict__ sg = P.s;
  const V *__restrict__ tg = P.t;
  const V *__restrict__ rh = P.rh;
  int64_t c0, c1;
  chunk_of(P.n, (int)gridDim.x, blockIdx.x, c0, c1);
  double acc[2] = {0.0, 0.0};
  for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBiUpd * kBlock) {
    V xv[kBiUpd], pv[kBiUpd], sv[kBiUpd], tv[kBiUpd], hv[kBiUpd];
#pragma unroll
    for (int u = 0; u < kBiUpd; ++u) {
      const int64_t i = g0 + (int64_t)u * kBlock;
      const bool in = i < c1;
      xv[u] = in ? x[i] : V(0);
      pv[u] = in ? p[i] : V(0);
      sv[u] = in ? sg[i] : V(0);
      tv[u] = (in && !ex) ? tg[i] : V(0);
      hv[u] = in ? rh[i] : V(0);
    }
#pragma unroll
    for (int u = 0; u < kBiUpd; ++u) {
      const int64_t i = g0 + (int64_t)u * kBlock;
      if (i < c1) {
        V ri;
        if (ex) {
          x[i] = fmav<V>(alpha, pv[u], xv[u]);
          ri = sv[u];
        } else {
          x[i] = fmav<V>(omega, sv[u], fmav<V>(alpha, pv[u], xv[u]));
          ri = fmav<V>(-omega, tv[u], sv[u]);
        }
        r[i] = ri;
        acc[0] = fma((double)hv[u], (double)ri, acc[0]);
        acc[1] = fma((double)ri, (double)ri, acc[1]);
      }
    }
  }
  block_sum<2>(acc);
  if (!publish_last<2>(acc, P.part, &P.C->ticket, (int)gridDim.x, blockIdx.x)) return;
  double tot[2];
  reduce_partials<2>(P.part, (int)gridDim.x, &P.C->ticket, tot);
  if (threadIdx.x != 0) return;
  BiCtl &C = *P.C;
  C.k += 1;
  if (C.exit_s) {
    C.rel = sqrt(C.ss) / C.nb;
    if (P.hist) P.hist[C.k] = C.rel;
    C.status = SLA_OK;
    C.done = 1;
    return;
  }
  const double rho_new = tot[0], rr = tot[1];
  C.rel = sqrt(rr) / C.nb;
  if (P.hist) P.hist[C.k] = C.rel;
  if (!isfinite(rr)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (sqrt(rr) <= C.rtol * C.nb) { C.status = SLA_OK; C.done = 1; return; }
  if (C.omega == 0.0) { C.status = SLA_BREAKDOWN; C.done = 1; return; }
  if (C.k >= C.maxit) { C.done = 1; return; }
  if (!isfinite(rho_new)) { C.status = SLA_NONFINITE; C.done = 1; return; }
  if (rho_new == 0.0) { C.status = SLA_BREAKDOWN; C.done = 1; return; }
  C.beta = (rho_new / C.rho) * (C.alpha / C.omega);
  C.rho = rho_new;
}

// ------------------------------------------------------------------------ resident engine
//
// The whole solve in one cooperative kernel: one 1024-thread block per SM owns a contiguous chunk of
// rows for the whole solve, the vectors live in global memory (in L2 at the sizes where the
// iteration count makes this matter), and the three global dependencies of an iteration (alpha
// needs rhat.v; the ||s|| test and omega need s.s, t.s, t.t; beta and the stopping test need
// rhat.r, r.r) are three grid barriers, each carrying a deterministic all-reduce: every block
// publishes its block sums, and after the barrier every block adds the G sums in the same fixed
// order, so all blocks hold bit-identical scalars and take the same branch.  In the products a
// column in the block's chunk reads the block's own p (or s); a column outside it recomputes
// p = r + beta (p_prev - omega v_prev) (or s = r - alpha v) from values the barrier published, read
// through L2 (another SM may hold a stale copy of them in its L1).  The barriers before omega and
// beta are split: while the other blocks arrive, a block forms x + alpha p and p - omega v, the
// parts of the next updates that need no pending scalar (each into a buffer free by then, with the
// roundings of the fused expressions).  Every barrier wait is bounded.
constexpr int kBrBlock = 1024;
constexpr int kBrVec = 4;   // rows per thread whose loads the p and s passes issue together
constexpr int kBrProd = 2;  // the product passes
constexpr int kBrUpd = 2;   // the update (five vectors per row)

// An all-reduce in two halves, so that a block can do work that needs neither side while the
// other blocks arrive: publish the block sums and arrive; then wait and form the grid totals
// (valid in warp 0).  The wait returns false when it expired; the solve then ends.
template <int NV>
__device__ __forceinline__ void br_publish_arrive(const double (&v)[NV], double *sbuf, double *part, int slot,
                                                  unsigned *arrive, unsigned &epoch) {
  block_publish<NV>(v, sbuf, part + (size_t)slot * kMaxBlocksPerSystem);
  grid_arrive(arrive, epoch);
}

template <int NV>
__device__ __forceinline__ bool br_wait_totals(const double *part, int slot, unsigned *arrive, unsigned *timeout,
                                               unsigned epoch, const WaitCfg &wc, double (&tot)[NV]) {
  if (!grid_wait(arrive, timeout, gridDim.x, epoch, wc)) return false;
  if (threadIdx.x < 32) warp_totals<NV>(part + (size_t)slot * kMaxBlocksPerSystem, (int)gridDim.x, tot);
  return true;
}

template <int NV>
__device__ __forceinline__ bool br_allreduce(const double (&v)[NV], double *sbuf, double *part, int slot,
                                             unsigned *arrive, unsigned *timeout, unsigned &epoch, const WaitCfg &wc,
                                             double (&tot)[NV]) {
  br_publish_arrive<NV>(v, sbuf, part, slot, arrive, epoch);
  return br_wait_totals<NV>(part, slot, arrive, timeout, epoch, wc, tot);
}

template <typename I>
__device__ __forceinline__ void br_row(const I *__restrict__ rp, int64_t i, int64_t nnz, uint32_t *bad, int64_t &e0,
                                       int64_t &e1) {
  e0 = (int64_t)rp[i];
  e1 = (int64_t)rp[i + 1];
  if (e0 < 0 || e1 < e0 || e1 > nnz) {
    atomicOr(bad, 1u);
    e0 = e1 = 0;
  }
}

// What thread 0 decides after a reduction and every thread of the block reads: the scalars of the
// next phase and whether the solve goes on.  The divisions and square roots run once per block
// (fp64 issue is this GPU's scarce resource; in 1024 threads they would cost a third of the rows'
// arithmetic).
struct BrScalars {
  double alpha, omega, beta;
  int go;      // 0: the solve ends here
  int exit_s;  // the ||s|| test passed: x += alpha p, r = s, then end
};

// Thread 0's solver state.
struct BrState {
  double nb, rho, alpha, omega, rel, rtol;
  int64_t k, maxit;
  int status;
};

template <typename V, typename I>
__global__ void __launch_bounds__(kBrBlock, 1) bi_resident(BiProb<V, I> P, WaitCfg wc) {
  __shared__ double sbuf[2 * kBrBlock];
  __shared__ BrScalars S;
  __shared__ BrState T;  // thread 0's solver state (identical in every block)
  BiCtl *C = P.C;
  unsigned *arrive = &C->arrive, *timeout = &C->timeout;
  uint32_t *bad = &C->bad;
  unsigned epoch = 0;
  const int64_t n = P.n, nnz = P.nnz;
  int64_t c0, c1;
  chunk_of(n, (int)gridDim.x, blockIdx.x, c0, c1);
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *__restrict__ val = P.val;
  V *__restrict__ x = P.x;
  V *__restrict__ r = P.r;
  V *__restrict__ rh = P.rh;
  V *__restrict__ sg = P.s;
  V *__restrict__ tg = P.t;
  const bool lead = threadIdx.x == 0;                    // decides for its block
  const bool hist = blockIdx.x == 0 && lead && P.hist;  // writes the history
  if (lead) {
    T.nb = T.rho = T.rel = 0.0;
    T.alpha = T.omega = 1.0;
    T.rtol = C->rtol;
    T.maxit = C->maxit;
    T.k = 0;
    T.status = SLA_NOT_CONVERGED;
  }

  // setup: x = x0 (or 0), r = b - A x0 (or b), rhat = r; ||b||^2 and r.r
  double a0[2] = {0.0, 0.0};
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kBrBlock) {
    const V bi = P.b[i];
    V ri = bi;
    if (P.x0) ri = bi - row_times(P, i, P.x0);
    const V xi = P.x0 ? P.x0[i] : V(0);
    r[i] = ri;
    rh[i] = ri;
    a0[0] = fma((double)bi, (double)bi, a0[0]);
    a0[1] = fma((double)ri, (double)ri, a0[1]);
    x[i] = xi;
  }
  double t0[2];
  const bool ok0 = br_allreduce<2>(a0, sbuf, P.part, 0, arrive, timeout, epoch, wc, t0);
  bool zero_x = false;
  if (lead) {
    S.go = 0;
    S.exit_s = 0;  // here: b = 0, x = 0 at the end
    S.beta = 0.0;
    if (ok0) {
      T.nb = sqrt(t0[0]);
      T.rho = t0[1];
      if (!isfinite(T.nb)) {
        T.status = SLA_NONFINITE;
      } else if (T.nb == 0.0) {
        S.exit_s = 1;
        T.status = SLA_OK;
        if (hist) P.hist[0] = 0.0;
      } else {
        T.rel = sqrt(t0[1]) / T.nb;
        if (hist) P.hist[0] = T.rel;
        if (!isfinite(t0[1])) T.status = SLA_NONFINITE;
        else if (sqrt(t0[1]) <= T.rtol * T.nb) T.status = SLA_OK;
        else if (T.maxit > 0) S.go = 1;
      }
    }
  }
  __syncthreads();
  zero_x = S.exit_s != 0;
  bool go = S.go != 0;
  V vbeta = V(0), vomega = V(1);
  int64_t kk = 0;  // every thread's iteration count
  while (go) {
    const int par = (int)(kk & 1);
    const bool first = kk == 0;
    const V *__restrict__ po = P.p[par ^ 1];
    const V *__restrict__ vo = P.v[par ^ 1];
    V *__restrict__ pn = P.p[par];
    V *__restrict__ vn = P.v[par];

    // p on the chunk's rows: r (first iteration) or r + beta w, with w = p_prev - omega v_prev
    // already in pn from the previous iteration's last wait (the same two roundings as p_at)
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrVec * kBrBlock) {
      V rv[kBrVec], wv[kBrVec];
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        const bool in = i < c1;
        rv[u] = in ? r[i] : V(0);
        wv[u] = (in && !first) ? pn[i] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) pn[i] = first ? rv[u] : fmav<V>(vbeta, wv[u], rv[u]);
      }
    }
    __syncthreads();
    // v = A p; rhat.v
    double a1[1] = {0.0};
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrProd * kBrBlock) {
      int64_t e0[kBrProd], e1[kBrProd];
      V hv[kBrProd];
#pragma unroll
      for (int u = 0; u < kBrProd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) {
          br_row<I>(rp, i, nnz, bad, e0[u], e1[u]);
          hv[u] = rh[i];
        } else {
          e0[u] = e1[u] = 0;
          hv[u] = V(0);
        }
      }
#pragma unroll
      for (int u = 0; u < kBrProd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i >= c1) continue;
        V a = V(0);
        for (int64_t e = e0[u]; e < e1[u]; ++e) {
          const int32_t c = ci[e];
          const V w = val[e];
          V pc;
          if ((int64_t)c >= c0 && (int64_t)c < c1) pc = pn[c];
          else if (col_ok(c, (int32_t)n, bad))
            pc = p_at<V>(__ldcg(r + c), first ? V(0) : __ldcg(po + c), first ? V(0) : __ldcg(vo + c), first, vbeta,
                         vomega);
          else pc = V(0);
          a = fmav<V>(w, pc, a);
        }
        vn[i] = a;
        a1[0] = fma((double)hv[u], (double)a, a1[0]);
      }
    }
    double t1[1];
    const bool ok1 = br_allreduce<1>(a1, sbuf, P.part, 2, arrive, timeout, epoch, wc, t1);
    if (lead) {
      S.go = 0;
      if (!ok1) {
      } else if (!isfinite(t1[0])) {
        T.status = SLA_NONFINITE;
      } else if (t1[0] == 0.0) {
        T.status = SLA_BREAKDOWN;
      } else {
        T.alpha = T.rho / t1[0];
        S.alpha = T.alpha;
        S.go = 1;
      }
    }
    __syncthreads();
    if (!S.go) break;
    const V valpha = (V)S.alpha;

    // s on the chunk's rows; s.s
    double a2[3] = {0.0, 0.0, 0.0};
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrVec * kBrBlock) {
      V rv[kBrVec], vv[kBrVec];
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        const bool in = i < c1;
        rv[u] = in ? r[i] : V(0);
        vv[u] = in ? vn[i] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) {
          const V si = fmav<V>(-valpha, vv[u], rv[u]);
          sg[i] = si;
          a2[0] = fma((double)si, (double)si, a2[0]);
        }
      }
    }
    __syncthreads();
    // t = A s; t.s, t.t
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrProd * kBrBlock) {
      int64_t e0[kBrProd], e1[kBrProd];
      V sv[kBrProd];
#pragma unroll
      for (int u = 0; u < kBrProd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) {
          br_row<I>(rp, i, nnz, bad, e0[u], e1[u]);
          sv[u] = sg[i];
        } else {
          e0[u] = e1[u] = 0;
          sv[u] = V(0);
        }
      }
#pragma unroll
      for (int u = 0; u < kBrProd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i >= c1) continue;
        V a = V(0);
        for (int64_t e = e0[u]; e < e1[u]; ++e) {
          const int32_t c = ci[e];
          const V w = val[e];
          V sc;
          if ((int64_t)c >= c0 && (int64_t)c < c1) sc = sg[c];
          else if (col_ok(c, (int32_t)n, bad)) sc = fmav<V>(-valpha, __ldcg(vn + c), __ldcg(r + c));
          else sc = V(0);
          a = fmav<V>(w, sc, a);
        }
        tg[i] = a;
        a2[1] = fma((double)a, (double)sv[u], a2[1]);
        a2[2] = fma((double)a, (double)a, a2[2]);
      }
    }
    double t2[3];
    br_publish_arrive<3>(a2, sbuf, P.part, 3, arrive, epoch);
    // while the other blocks arrive: xh = x + alpha p, the part of the x update that does not need
    // omega, into v_prev's buffer (every block read v_prev before the last barrier); x itself
    // stays the last iterate until the update
    V *__restrict__ xh = P.v[par ^ 1];
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrVec * kBrBlock) {
      V xv[kBrVec], pv[kBrVec];
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        const bool in = i < c1;
        xv[u] = in ? x[i] : V(0);
        pv[u] = in ? pn[i] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kBrVec; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) xh[i] = fmav<V>(valpha, pv[u], xv[u]);
      }
    }
    const bool ok2 = br_wait_totals<3>(P.part, 3, arrive, timeout, epoch, wc, t2);
    if (lead) {
      S.go = 0;
      S.exit_s = 0;
      if (!ok2) {
      } else if (!isfinite(t2[0])) {
        T.status = SLA_NONFINITE;
      } else if (sqrt(t2[0]) <= T.rtol * T.nb) {
        S.exit_s = 1;  // x += alpha p, r = s; the solve ends after the update
        T.rel = sqrt(t2[0]) / T.nb;
        T.status = SLA_OK;
      } else if (!isfinite(t2[1]) || !isfinite(t2[2])) {
        T.status = SLA_NONFINITE;
      } else if (t2[2] == 0.0) {
        T.status = SLA_BREAKDOWN;
      } else {
        T.omega = t2[1] / t2[2];
        S.omega = T.omega;
        S.go = 1;
      }
    }
    __syncthreads();
    const bool exit_s = S.exit_s != 0;
    if (!S.go && !exit_s) break;
    const V vom = exit_s ? V(0) : (V)S.omega;

    // x = xh + omega s, r = s - omega t (x = xh, r = s after the early test); rhat.r, r.r
    double a3[2] = {0.0, 0.0};
    for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrUpd * kBrBlock) {
      V xv[kBrUpd], sv[kBrUpd], tv[kBrUpd], hv[kBrUpd];
#pragma unroll
      for (int u = 0; u < kBrUpd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        const bool in = i < c1;
        xv[u] = in ? xh[i] : V(0);
        sv[u] = in ? sg[i] : V(0);
        tv[u] = (in && !exit_s) ? tg[i] : V(0);
        hv[u] = in ? rh[i] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kBrUpd; ++u) {
        const int64_t i = g0 + (int64_t)u * kBrBlock;
        if (i < c1) {
          V ri;
          if (exit_s) {
            x[i] = xv[u];
            ri = sv[u];
          } else {
            x[i] = fmav<V>(vom, sv[u], xv[u]);
            ri = fmav<V>(-vom, tv[u], sv[u]);
          }
          r[i] = ri;
          a3[0] = fma((double)hv[u], (double)ri, a3[0]);
          a3[1] = fma((double)ri, (double)ri, a3[1]);
        }
      }
    }
    kk += 1;
    if (exit_s) {
      if (lead) {
        T.k = kk;
        if (hist) P.hist[kk] = T.rel;
      }
      break;
    }
    double t3[2];
    br_publish_arrive<2>(a3, sbuf, P.part, 6, arrive, epoch);
    // while the other blocks arrive: w = p - omega v, the part of the next p that does not need
    // beta, into p_prev's buffer (the next iteration's p; every block read p_prev before the first
    // barrier of this iteration).  Wasted if the solve stops here.
    {
      V *__restrict__ wn = P.p[par ^ 1];
      for (int64_t g0 = c0 + threadIdx.x; g0 < c1; g0 += (int64_t)kBrVec * kBrBlock) {
        V pv[kBrVec], vv[kBrVec];
#pragma unroll
        for (int u = 0; u < kBrVec; ++u) {
          const int64_t i = g0 + (int64_t)u * kBrBlock;
          const bool in = i < c1;
          pv[u] = in ? pn[i] : V(0);
          vv[u] = in ? vn[i] : V(0);
        }
#pragma unroll
        for (int u = 0; u < kBrVec; ++u) {
          const int64_t i = g0 + (int64_t)u * kBrBlock;
          if (i < c1) wn[i] = fmav<V>(-vom, vv[u], pv[u]);
        }
      }
    }
    const bool ok3 = br_wait_totals<2>(P.part, 6, arrive, timeout, epoch, wc, t3);
    if (lead) {
      S.go = 0;
      if (ok3) {
        T.k = kk;
        T.rel = sqrt(t3[1]) / T.nb;
        if (hist) P.hist[kk] = T.rel;
        if (!isfinite(t3[1])) T.status = SLA_NONFINITE;
        else if (sqrt(t3[1]) <= T.rtol * T.nb) T.status = SLA_OK;
        else if (T.omega == 0.0) T.status = SLA_BREAKDOWN;
        else if (kk >= T.maxit) {
        } else if (!isfinite(t3[0])) T.status = SLA_NONFINITE;
        else if (t3[0] == 0.0) T.status = SLA_BREAKDOWN;
        else {
          const double beta = (t3[0] / T.rho) * (T.alpha / T.omega);
          T.rho = t3[0];
          S.beta = beta;
          S.go = 1;
        }
      }
    }
    __syncthreads();
    if (!S.go) break;
    vbeta = (V)S.beta;
    vomega = vom;
  }
  if (zero_x)
    for (int64_t i = c0 + threadIdx.x; i < c1; i += kBrBlock) x[i] = V(0);
  if (blockIdx.x == 0 && lead) {
    C->k = T.k;
    C->rel = T.rel;
    C->status = T.status;
    C->done = 1;
  }
}

// Blocks of the resident kernel: one per SM, each with at least 256 rows; 0 when it cannot run
// (no co-residency, or a barrier count past the 32-bit counter).
template <typename V, typename I>
int br_grid(int64_t n, int64_t maxit) {
  int dev = 0, sms = 0, per_sm = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (!coop ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bi_resident<V, I>, kBrBlock, 0) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return 0;
  }
  int64_t g = (n + 255) / 256;
  if (g > sms) g = sms;
  if (g > kMaxBlocksPerSystem) g = kMaxBlocksPerSystem;
  if (g < 1) g = 1;
  if ((double)(3 * maxit + 2) * (double)g >= 4.0e9) return 0;
  return (int)g;
}

// x = 0 when b = 0.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) bi_finish(BiProb<V, I> P) {
  if (!P.C->zero_x) return;
  BI_ROWS(i) P.x[i] = V(0);
}

// vt[e] = val[e'] for the entry e' = (j, i) partnering e = (i, j): A^T's values on A's pattern when
// the pattern is structurally symmetric (columns sorted within rows).  A missing partner sets
// `nopartner` (A^T is then built explicitly); a malformed row range or column sets `bad`.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) bi_transpose_values(int64_t n, int64_t nnz, const I *__restrict__ rp,
                                                              const int32_t *__restrict__ ci,
                                                              const V *__restrict__ val, V *__restrict__ vt,
                                                              uint32_t *bad, uint32_t *nopartner) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock) {
    int64_t e0, e1;
    row_range(rp, i, nnz, e0, e1, bad);
    for (int64_t e = e0; e < e1; ++e) {
      const int32_t j = ci[e];
      V out = V(0);
      bool found = false;
      const bool jok = col_ok(j, (int32_t)n, bad);
      if (jok) {
        int64_t j0, j1;
        row_range(rp, j, nnz, j0, j1, bad);
        int64_t lo = j0, hi = j1;
        while (lo < hi) {  // the first entry of row j with column >= i (columns sorted per row)
          const int64_t mid = lo + (hi - lo) / 2;
          if (ci[mid] < i) lo = mid + 1;
          else hi = mid;
        }
        if (lo < j1 && ci[lo] == (int32_t)i) {
          out = val[lo];
          found = true;
        }
      }
      if (jok && !found) atomicOr(nopartner, 1u);
      vt[e] = out;
    }
  }
}

// ---- explicit A^T for patterns without partner entries (run only on a well-formed CSR)
//
// Column counts, an exclusive scan of them into A^T's row pointers (per-chunk sums, a scan of the
// chunk sums, per-chunk scans), a scatter through per-column cursors, and a sort of every A^T row
// by column: the scatter's order depends on the atomics' timing, the sorted rows do not (given no
// duplicate entries), so the adjoint solve sums every row of A^T in the same order each time.

template <typename I>
__global__ void __launch_bounds__(kBlock) tr_count(int64_t n, const I *__restrict__ rp, const int32_t *__restrict__ ci,
                                                   int32_t *cnt) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock)
    for (int64_t e = (int64_t)rp[i]; e < (int64_t)rp[i + 1]; ++e) atomicAdd(cnt + ci[e], 1);
}

// Block sum of one int64 per thread of a 1024-thread block, in thread 0.
__device__ __forceinline__ int64_t tr_block_sum(int64_t v, int64_t *s_w) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = v;
  __syncthreads();
  int64_t t = 0;
  if (threadIdx.x < 32) {
    t = s_w[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
  }
  __syncthreads();
  return t;
}

// Exclusive scan of one int64 per thread of a 1024-thread block; every thread gets its prefix.
__device__ __forceinline__ int64_t tr_block_exscan(int64_t v, int64_t *s_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int64_t w = s_w[lane], winc = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += y;
    }
    s_w[lane] = winc - w;  // exclusive prefix of the warp sums
  }
  __syncthreads();
  const int64_t out = s_w[warp] + inc - v;
  __syncthreads();
  return out;
}

// bsum[b] = sum of cnt over chunk b (kTrChunk rows: 1024 threads x 4).
__global__ void __launch_bounds__(1024) tr_chunk_sums(int64_t n, const int32_t *__restrict__ cnt, int64_t *bsum) {
  __shared__ int64_t s_w[32];
  const int64_t base = blockIdx.x * kTrChunk + (int64_t)threadIdx.x * 4;
  int64_t v = 0;
  for (int u = 0; u < 4; ++u)
    if (base + u < n) v += cnt[base + u];
  const int64_t t = tr_block_sum(v, s_w);
  if (threadIdx.x == 0) bsum[blockIdx.x] = t;
}

// bsum[0..nb) replaced by its exclusive scan, and bsum[nb] = the total; one block.
__global__ void __launch_bounds__(1024) tr_scan_sums(int64_t nb, int64_t *bsum) {
  __shared__ int64_t s_w[32];
  const int64_t per = (nb + 1023) / 1024;
  const int64_t a = (int64_t)threadIdx.x * per, b = a + per < nb ? a + per : nb;
  int64_t v = 0;
  for (int64_t k = a; k < b; ++k) v += bsum[k];
  int64_t run = tr_block_exscan(v, s_w);
  __syncthreads();
  for (int64_t k = a; k < b; ++k) {
    const int64_t c = bsum[k];
    bsum[k] = run;
    run += c;
  }
  if (b == nb && a < b) bsum[nb] = run;  // the thread holding the last chunk
  if (nb == 0 && threadIdx.x == 0) bsum[0] = 0;
}

// tp[j] = bsum[chunk] + the exclusive prefix of cnt within the chunk; tp[n] = the total.
template <typename I>
__global__ void __launch_bounds__(1024) tr_chunk_scan(int64_t n, const int32_t *__restrict__ cnt,
                                                      const int64_t *__restrict__ bsum, I *tp) {
  __shared__ int64_t s_w[32];
  const int64_t base = blockIdx.x * kTrChunk + (int64_t)threadIdx.x * 4;
  int64_t c[4], v = 0;
  for (int u = 0; u < 4; ++u) {
    c[u] = base + u < n ? cnt[base + u] : 0;
    v += c[u];
  }
  int64_t run = bsum[blockIdx.x] + tr_block_exscan(v, s_w);
  for (int u = 0; u < 4; ++u) {
    if (base + u < n) tp[base + u] = (I)run;
    run += c[u];
    if (base + u == n - 1) tp[n] = (I)run;
  }
}

// Scatter every entry (i, j) of A into row j of A^T through the column's cursor.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) tr_scatter(int64_t n, const I *__restrict__ rp, const int32_t *__restrict__ ci,
                                                     const V *__restrict__ val, const I *__restrict__ tp,
                                                     int32_t *cur, int32_t *__restrict__ tci, V *__restrict__ tval) {
  for (int64_t i = blockIdx.x * (int64_t)kBlock + threadIdx.x; i < n; i += (int64_t)gridDim.x * kBlock)
    for (int64_t e = (int64_t)rp[i]; e < (int64_t)rp[i + 1]; ++e) {
      const int32_t j = ci[e];
      const int64_t pos = (int64_t)tp[j] + atomicAdd(cur + j, 1);
      tci[pos] = (int32_t)i;
      tval[pos] = val[e];
    }
}

// Sort every row of A^T by column (insertion sort, one thread per row), values alongside.
template <typename V, typename I>
__global__ void __launch_bounds__(kBlock) tr_sort_rows(int64_t n, const I *__restrict__ tp, int32_t *__restrict__ tci,
                                                       V *__restrict__ tval) {
  for (int64_t j = blockIdx.x * (int64_t)kBlock + threadIdx.x; j < n; j += (int64_t)gridDim.x * kBlock) {
    const int64_t a = (int64_t)tp[j], b = (int64_t)tp[j + 1];
    for (int64_t k = a + 1; k < b; ++k) {
      const int32_t key = tci[k];
      const V kv = tval[k];
      int64_t m = k - 1;
      while (m >= a && tci[m] > key) {
        tci[m + 1] = tci[m];
        tval[m + 1] = tval[m];
        --m;
      }
      tci[m + 1] = key;
      tval[m + 1] = kv;
    }
  }
}

// Builds A^T (row pointers tp of A's index type, columns tci, values tval) from a well-formed A.
template <typename V, typename I>
sla_status tr_build(const sla_csr *A, const BiLayout &L, char *ws, cudaStream_t st) {
  const int64_t n = A->n;
  int32_t *cnt = (int32_t *)(ws + L.cnt);
  int64_t *bsum = (int64_t *)(ws + L.bsum);
  I *tp = (I *)(ws + L.tp);
  const I *rp = (const I *)A->row_ptr;
  const int G = bi_grid(n);
  const int64_t nb = (n + kTrChunk - 1) / kTrChunk;
  cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (size_t)n, st);
  if (e != cudaSuccess) return fail(e);
  tr_count<I><<<G, kBlock, 0, st>>>(n, rp, A->col_idx, cnt);
  tr_chunk_sums<<<(unsigned)nb, 1024, 0, st>>>(n, cnt, bsum);
  tr_scan_sums<<<1, 1024, 0, st>>>(nb, bsum);
  tr_chunk_scan<I><<<(unsigned)nb, 1024, 0, st>>>(n, cnt, bsum, tp);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
  if ((e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (size_t)n, st)) != cudaSuccess) return fail(e);
  tr_scatter<V, I><<<G, kBlock, 0, st>>>(n, rp, A->col_idx, (const V *)A->values, tp, cnt, (int32_t *)(ws + L.tci),
                                         (V *)(ws + L.vt));
  tr_sort_rows<V, I><<<G, kBlock, 0, st>>>(n, tp, (int32_t *)(ws + L.tci), (V *)(ws + L.vt));
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
  count_launches(6);
  return SLA_OK;
}

// The resident engine: one cooperative launch for the whole solve.  SLA_INVALID_ARG when it cannot
// be launched here (the caller then runs the host loop); the control block is already initialised.
template <typename V, typename I>
sla_status bi_run_resident(BiProb<V, I> P, int G, cudaStream_t st, sla_cg_info *info) {
  WaitCfg wc = launch_wait_cfg();
  void *args[] = {(void *)&P, (void *)&wc};
  cudaError_t e = cudaLaunchCooperativeKernel((void *)bi_resident<V, I>, dim3(G), dim3(kBrBlock), args, 0, st);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();  // refused before anything ran
    return SLA_INVALID_ARG;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  count_launches(1);
  BiCtl h;
  if ((e = cudaMemcpyAsync(&h, P.C, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
  if (info) {
    info->iters = h.k;
    info->rel_res = h.rel;
    info->status = h.timeout ? SLA_TIMEOUT : h.bad ? SLA_BAD_CSR : (sla_status)h.status;
    info->kernels = 1;
    info->path = SLA_LOOP_RESIDENT;
  }
  return SLA_OK;
}

template <typename V, typename I>
sla_status bi_run(BiProb<V, I> P, const sla_cg_opts *o, cudaStream_t st, sla_cg_info *info) {
  const int G = bi_grid(P.n), Gu = bi_upd_grid(P.n);
  BiCtl init;
  memset(&init, 0, sizeof(init));
  init.maxit = o->maxit;
  init.rtol = o->rtol;
  cudaError_t e = cudaMemcpyAsync(P.C, &init, sizeof(init), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(e);
  if (o->loop != SLA_LOOP_HOST) {
    const int Gr = br_grid<V, I>(P.n, o->maxit);
    if (Gr > 0) {
      const sla_status s = bi_run_resident<V, I>(P, Gr, st, info);
      if (s != SLA_INVALID_ARG) return s;
    }
  }
  uint64_t launches = 0;
  bi_setup<V, I><<<G, kBlock, 0, st>>>(P);
  ++launches;
  const int64_t U = o->unroll > 0 ? o->unroll : 8;
  BiCtl h;
  memset(&h, 0, sizeof(h));
  for (int64_t k = 0; k < o->maxit; k += U) {
    const int64_t upto = (o->maxit - k) < U ? (o->maxit - k) : U;
    for (int64_t u = 0; u < upto; ++u) {
      bi_dir_apply<V, I><<<G, kBlock, 0, st>>>(P);
      bi_s_apply<V, I><<<G, kBlock, 0, st>>>(P);
      bi_update<V, I><<<Gu, kBlock, 0, st>>>(P);
    }
    launches += 3 * (uint64_t)upto;
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    if ((e = cudaMemcpyAsync(&h, P.C, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
    if (h.done) break;
  }
  bi_finish<V, I><<<G, kBlock, 0, st>>>(P);
  ++launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
  if ((e = cudaMemcpyAsync(&h, P.C, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
  count_launches(launches);
  if (info) {
    info->iters = h.k;
    info->rel_res = h.rel;
    info->status = h.bad ? SLA_BAD_CSR : (sla_status)h.status;
    info->kernels = (int64_t)launches;
    info->path = SLA_LOOP_HOST;
  }
  return SLA_OK;
}

template <typename V, typename I>
BiProb<V, I> bi_prob(const sla_csr *A, const void *values, const void *b, const void *x0, void *x, double *hist,
                     char *ws) {
  const BiLayout L = bi_layout(A->n, A->nnz, sizeof(V));
  BiProb<V, I> P;
  P.n = A->n;
  P.nnz = A->nnz;
  P.rp = (const I *)A->row_ptr;
  P.ci = A->col_idx;
  P.val = (const V *)values;
  P.b = (const V *)b;
  P.x0 = (const V *)x0;
  P.x = (V *)x;
  P.r = (V *)(ws + L.r);
  P.rh = (V *)(ws + L.rh);
  for (int j = 0; j < 2; ++j) {
    P.p[j] = (V *)(ws + L.p[j]);
    P.v[j] = (V *)(ws + L.v[j]);
  }
  P.s = (V *)(ws + L.s);
  P.t = (V *)(ws + L.t);
  P.part = (double *)(ws + L.part);
  P.hist = hist;
  P.C = (BiCtl *)(ws + L.ctl);
  return P;
}

bool bi_opts_ok(const sla_cg_opts *o) {
  return check_opts(o) == SLA_OK && o->precond == SLA_PRECOND_NONE;
}

template <typename V, typename I>
sla_status bi_solve_t(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *o, void *x,
                      sla_cg_info *info, double *hist, char *ws, cudaStream_t st) {
  return bi_run<V, I>(bi_prob<V, I>(A, A->values, b, x0, x, hist, ws), o, st, info);
}

template <typename V, typename I>
sla_status bi_adjoint_t(const sla_csr *A, const void *x, const void *g, const sla_cg_opts *o, void *grad_b,
                        void *grad_values, sla_cg_info *info, char *ws, cudaStream_t st) {
  const BiLayout L = bi_layout(A->n, A->nnz, sizeof(V));
  BiProb<V, I> P = bi_prob<V, I>(A, ws + L.vt, g, nullptr, grad_b, nullptr, ws);
  // the control block is cleared first so that the transpose's bad flag starts at 0; the flag is
  // read before the solve, whose own start clears the block again
  BiCtl init;
  memset(&init, 0, sizeof(init));
  cudaError_t e = cudaMemcpyAsync(P.C, &init, sizeof(init), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(e);
  const int G = bi_grid(A->n);
  bi_transpose_values<V, I><<<G, kBlock, 0, st>>>(A->n, A->nnz, (const I *)A->row_ptr, A->col_idx,
                                                   (const V *)A->values, (V *)(ws + L.vt), &P.C->bad,
                                                   &P.C->nopartner);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
  count_launches(1);
  BiCtl h;
  if ((e = cudaMemcpyAsync(&h, P.C, sizeof(h), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return fail(e);
  if (h.bad) {
    if (info) {
      memset(info, 0, sizeof(*info));
      info->status = SLA_BAD_CSR;
      info->path = SLA_LOOP_HOST;
    }
    return SLA_OK;
  }
  if (h.nopartner) {
    // the pattern is not structurally symmetric: solve on an explicitly built A^T
    SLA_CHECK((tr_build<V, I>(A, L, ws, st)));
    P.rp = (const I *)(ws + L.tp);
    P.ci = (const int32_t *)(ws + L.tci);
  }
  sla_status s = bi_run<V, I>(P, o, st, info);
  if (s != SLA_OK) return s;
  if (grad_values) SLA_CHECK(grad_values_entry(A, 1, grad_b, x, grad_values, st));
  return SLA_OK;
}

}  // namespace
}  // namespace sla

using namespace sla;

extern "C" {

size_t sla_bicgstab_workspace_bytes(int64_t n, int64_t nnz, int32_t dtype) {
  if (n < 0 || nnz < 0 || (dtype != SLA_F32 && dtype != SLA_F64)) return 0;
  return bi_layout(n, nnz, dtype == SLA_F64 ? 8 : 4).total;
}

sla_status sla_bicgstab_solve(const sla_csr *A, const void *b, const void *x0, const sla_cg_opts *opts, void *x,
                              sla_cg_info *info, double *history, void *workspace, size_t ws_bytes, void *stream) {
  SLA_CHECK(check_csr(A, true));
  if (!bi_opts_ok(opts)) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(b, A, false));
  SLA_CHECK(check_vec(x0, A, true));
  SLA_CHECK(check_vec(x, A, false));
  if (history && !aligned(history, 8)) return SLA_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return SLA_INVALID_ARG;
  if (ws_bytes < bi_layout(A->n, A->nnz, A->dtype == SLA_F64 ? 8 : 4).total) return SLA_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  if (A->n == 0) {
    if (info) {
      memset(info, 0, sizeof(*info));
      info->path = SLA_LOOP_HOST;
    }
    if (history) {
      cudaError_t e = cudaMemsetAsync(history, 0, sizeof(double), st);
      if (e != cudaSuccess) return fail(e);
    }
    return SLA_OK;
  }
  char *ws = (char *)workspace;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64) return bi_solve_t<double, int64_t>(A, b, x0, opts, x, info, history, ws, st);
    return bi_solve_t<double, int32_t>(A, b, x0, opts, x, info, history, ws, st);
  }
  if (A->rowptr_type == SLA_I64) return bi_solve_t<float, int64_t>(A, b, x0, opts, x, info, history, ws, st);
  return bi_solve_t<float, int32_t>(A, b, x0, opts, x, info, history, ws, st);
}

sla_status sla_bicgstab_adjoint(const sla_csr *A, const void *x, const void *g, const sla_cg_opts *opts,
                                void *grad_b, void *grad_values, sla_cg_info *info, void *workspace, size_t ws_bytes,
                                void *stream) {
  SLA_CHECK(check_csr(A, true));
  if (!bi_opts_ok(opts)) return SLA_INVALID_ARG;
  SLA_CHECK(check_vec(x, A, false));
  SLA_CHECK(check_vec(g, A, false));
  SLA_CHECK(check_vec(grad_b, A, false));
  SLA_CHECK(check_vec(grad_values, A, true));
  if (!workspace || !aligned(workspace, 256)) return SLA_INVALID_ARG;
  if (ws_bytes < bi_layout(A->n, A->nnz, A->dtype == SLA_F64 ? 8 : 4).total) return SLA_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  if (A->n == 0) {
    if (info) {
      memset(info, 0, sizeof(*info));
      info->path = SLA_LOOP_HOST;
    }
    return SLA_OK;
  }
  char *ws = (char *)workspace;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64)
      return bi_adjoint_t<double, int64_t>(A, x, g, opts, grad_b, grad_values, info, ws, st);
    return bi_adjoint_t<double, int32_t>(A, x, g, opts, grad_b, grad_values, info, ws, st);
  }
  if (A->rowptr_type == SLA_I64) return bi_adjoint_t<float, int64_t>(A, x, g, opts, grad_b, grad_values, info, ws, st);
  return bi_adjoint_t<float, int32_t>(A, x, g, opts, grad_b, grad_values, info, ws, st);
}

}  // extern "C"
