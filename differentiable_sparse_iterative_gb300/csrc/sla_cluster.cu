// Cluster-resident CG: the whole solve of each system of a batch in one thread-block cluster.
//
// Method as in sla_cg.cu ("torch-sla" technical summary, Methodology 1-2 and Significance:
// Hestenes-Stiefel CG with optional Jacobi preconditioning; same recurrences, same stopping
// rule, same status decisions).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "sla_common.cuh"
#include "sla_host.h"
#include "sla_onchip.cuh"

namespace sla {

namespace {

// ---------------------------------------------------------------- cluster-resident kernel
//
// One thread-block cluster of C CTAs (C <= 16) solves one system; a batch is a grid of clusters.
// CTA j of a cluster keeps x, r, p, q (and 1/diag) of its row chunk in shared memory for the whole
// solve; nothing goes through global memory during the iteration except the matrix stream.  When
// shared memory has room for a second p buffer (two_p), p_k is written to buffer k & 1 while the
// partners still read p_{k-1} from the other, and p_k of a row owned by a partner CTA is formed
// from the partner's r_k (1/diag) and p_{k-1}, read from its shared memory (distributed shared
// memory) with the partner's own expression, so the same bits: the two dependencies of an
// iteration (p.q and r.r) are then the only hardware cluster barriers.  Otherwise p of a
// partner's row is read from the partner's shared memory once a third barrier has made every
// CTA's p_k visible.  Each all-reduce adds the C block sums in rank order in every CTA, so all
// CTAs of a cluster hold bit-identical scalars.
namespace cgs = cooperative_groups;
constexpr int kClBlock = 256;
constexpr int kClMax = 16;
constexpr size_t kClSmemMax = 110 * 1024;  // dynamic shared memory a cluster CTA may use
#ifndef SLA_CLUSTER_ROWS
#define SLA_CLUSTER_ROWS 1
#endif
#ifndef SLA_CLUSTER_ENTRIES
#define SLA_CLUSTER_ENTRIES 5
#endif
#ifndef SLA_CLUSTER_STAGE_RO
#define SLA_CLUSTER_STAGE_RO 1
#endif
constexpr int kClR = SLA_CLUSTER_ROWS;     // rows per thread whose entries the streamed SpMV loads together
constexpr int kClK = SLA_CLUSTER_ENTRIES;  // entries per row loaded up front (the rest one by one)
constexpr int kClGroup = 8;  // rows per thread whose p.q and r.r terms are summed in the data type

// Sum of the C partners' value slot[q] (read through distributed shared memory), for warp 0:
// lane j reads partner j, then a log2(C)-level shuffle tree (C is a power of two); every CTA of
// the cluster obtains the same bits.  Result valid in lane 0.  Each fp64 add costs a warp 64
// cycles of its sub-partition's fp64 unit on this GPU, so the tree has no more levels than C needs.
template <int NQ>
__device__ __forceinline__ void cluster_sum(cgs::cluster_group &cl, double *slot, int C, double (&out)[NQ]) {
  const int lane = threadIdx.x & 31;
  double v[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) v[q] = 0.0;
  if (lane < C) {
    const double *ps = cl.map_shared_rank(slot, lane);
#pragma unroll
    for (int q = 0; q < NQ; ++q) v[q] = ps[q];
  }
  for (int o = C >> 1; o > 0; o >>= 1)
#pragma unroll
    for (int q = 0; q < NQ; ++q) v[q] += __shfl_down_sync(0xffffffffu, v[q], o);
#pragma unroll
  for (int q = 0; q < NQ; ++q) out[q] = v[q];
}

// Block sum of NV values per thread, result in thread 0, in a fixed order.  Warps 0-3 (one per SM
// sub-partition, so their fp64 adds run in parallel) each add CB/4 values: a pairwise tree over
// the CB/128 values of a lane, then a shuffle tree; thread 0 adds the four warp sums.
// sb: shared scratch of NV * CB doubles.
template <int NV, int CB>
__device__ __forceinline__ void block_sum4(double (&v)[NV], double *sb) {
  static_assert(CB % 128 == 0 && CB <= 1024, "block of 128..1024 threads");
  constexpr int PER = CB / 128;
  __shared__ double s4[NV][4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int j = 0; j < NV; ++j) sb[j * CB + tid] = v[j];
  __syncthreads();
  if (warp < 4) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      double a[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) a[u] = sb[j * CB + warp * (CB / 4) + lane + 32 * u];
#pragma unroll
      for (int w = 1; w < PER; w <<= 1)
#pragma unroll
        for (int u = 0; u + w < PER; u += 2 * w) a[u] += a[u + w];
      const double t = warp_sum(a[0]);
      if (lane == 0) s4[j][warp] = t;
    }
  }
  __syncthreads();
  if (tid == 0)
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = (s4[j][0] + s4[j][1]) + (s4[j][2] + s4[j][3]);
}

template <typename V, typename I, bool JAC, int CB>
__global__ void __launch_bounds__(CB) cg_cluster(Prob<V, I> P, int C, int cap, int mcap, int ro_on, int two_p) {
  cgs::cluster_group cl = cgs::this_cluster();
  const int rank = (int)cl.block_rank();
  const int sys = (int)(blockIdx.x / (unsigned)C);
  const int tid = threadIdx.x;
  extern __shared__ __align__(16) unsigned char smem_cl[];
  // x, r, p (two buffers with two_p), q (and 1/diag), cap rows each, in this order in every CTA
  V *sx = reinterpret_cast<V *>(smem_cl);
  V *sr = sx + cap;
  V *sp0 = sr + cap;
  V *sp1 = two_p ? sp0 + cap : sp0;
  V *sq = sp1 + cap;
  V *sd = JAC ? sq + cap : nullptr;
  const int64_t sq_off = (int64_t)(two_p ? 4 : 3) * cap;  // offsets of q and 1/diag in every CTA's layout
  // optional copy of the CTA's CSR slice (mcap > 0): row offsets, columns, values; or of its row
  // offsets alone (ro_on)
  int32_t *s_ro = reinterpret_cast<int32_t *>(sq + cap + (JAC ? cap : 0));
  int32_t *s_ci = s_ro + ((cap + 1 + 3) & ~3);  // padded so the values below stay 16-byte aligned
  V *s_val = reinterpret_cast<V *>(s_ci + ((mcap + 3) & ~3));
  __shared__ double s_part[2][5];  // [0]: setup sums, then r.r / r.z; [1]: p.q (partners read these)
  // block-sum scratch for two values per thread: the iterations sum at most two; the five setup
  // sums go through it in three passes.  (Five values' worth, 20 KB at 512 threads, kept two
  // CTAs with a second p buffer from sharing an SM.)
  __shared__ double s_red[2 * CB];
  __shared__ V *s_peer[kClMax];    // partners' vectors (the address of their x) in distributed shared memory
  __shared__ int32_t s_start[kClMax + 1];  // first row of each partner (n for the end)
  // beta, alpha, alpha_prev in the data type, converted once by thread 0 (a conversion is an fp64
  // instruction, 64 cycles of a sub-partition's fp64 unit, if every warp made its own)
  __shared__ V s_vsc[3];
  __shared__ ResScalars S;
  __shared__ int s_pending;

  const int64_t n = P.n;
  auto start_of = [&](int j) { return n * j / C; };
  const int64_t c0 = start_of(rank), c1 = start_of(rank + 1);
  const int len = (int)(c1 - c0);
  const int64_t vo = (int64_t)sys * n;
  const V *__restrict__ val = P.val + (int64_t)sys * P.val_stride;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *b = P.b + vo;
  const V *x0 = P.x0 ? P.x0 + vo : nullptr;
  V *xg = P.x + vo;
  double *hist = P.history ? P.history + (size_t)sys * (size_t)(P.maxit + 1) : nullptr;
  Ctl *Cs = P.ctl + sys;
  Glob *glob = P.glob;
  if (tid < C) s_peer[tid] = cl.map_shared_rank(sx, tid);
  if (tid <= C) s_start[tid] = (int32_t)start_of(tid);
  if (blockIdx.x == 0 && tid == 0) atomicAdd(&glob->kernels, 1ull);

  // ---- setup
  double acc5[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
  for (int li = tid; li < len; li += CB) {
    const int64_t i = c0 + li;
    int64_t e0, e1;
    row_range(rp, i, P.nnz, e0, e1, &glob->bad_csr);
    const V bi = b[i];
    V ri = bi;
    if (x0) {
      V s_ = V(0);
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = ci[e];
        if (col_ok(c, (int32_t)n, &glob->bad_csr)) s_ = fmav<V>(val[e], x0[c], s_);
      }
      ri = bi - s_;
      sx[li] = x0[i];
    } else {
      sx[li] = V(0);
    }
    sr[li] = ri;
    acc5[0] = fma((double)bi, (double)bi, acc5[0]);
    acc5[1] = fma((double)ri, (double)ri, acc5[1]);
    if (JAC) {
      V d = V(0);
      for (int64_t e = e0; e < e1; ++e)
        if (ci[e] == (int32_t)i) d = val[e];
      if (!isfinite((double)d)) acc5[3] += 1.0;
      else if (!(d > V(0))) acc5[4] += 1.0;
      const V di = V(1) / d;
      sd[li] = di;
      acc5[2] = fma((double)ri, (double)(di * ri), acc5[2]);
    }
  }
  // the matrix does not change during the solve: keep the CTA's slice on chip when it fits
  const int64_t m_lo = len > 0 ? (int64_t)rp[c0] : 0, m_hi = len > 0 ? (int64_t)rp[c1] : 0;
  const bool slice_ok = m_lo >= 0 && m_hi >= m_lo && m_hi <= P.nnz && (m_hi - m_lo) < (int64_t)INT32_MAX;
  const bool mstaged = mcap > 0 && slice_ok && (m_hi - m_lo) <= mcap;
  const bool rostaged = mstaged || (ro_on && slice_ok);
  if (rostaged) {
    // offsets relative to the slice, clamped into it: a malformed row_ptr is reported and can
    // never index outside the slice
    const int64_t mlen = m_hi - m_lo;
    for (int li = tid; li <= len; li += CB) {
      int64_t o = (int64_t)rp[c0 + li] - m_lo;
      if (o < 0 || o > mlen) {
        atomicOr(&glob->bad_csr, 1u);
        o = o < 0 ? 0 : mlen;
      }
      s_ro[li] = (int32_t)o;
    }
  }
  if (mstaged) {
    for (int64_t e = m_lo + tid; e < m_hi; e += CB) {
      s_ci[e - m_lo] = ci[e];
      s_val[e - m_lo] = val[e];
    }
  }
  {
    double a01[2] = {acc5[0], acc5[1]}, a23[2] = {acc5[2], acc5[3]}, a4[1] = {acc5[4]};
    block_sum4<2, CB>(a01, s_red);
    block_sum4<2, CB>(a23, s_red);
    block_sum4<1, CB>(a4, s_red);
    acc5[0] = a01[0];
    acc5[1] = a01[1];
    acc5[2] = a23[0];
    acc5[3] = a23[1];
    acc5[4] = a4[0];
  }
  if (tid == 0)
    for (int q = 0; q < 5; ++q) s_part[0][q] = acc5[q];
  cl.sync();
  int status = SLA_NOT_CONVERGED, pending = 0;
  int64_t k = 0;
  double rel = 0.0, rr_last = -1.0;
  double t5[5];
  if (tid < 32) cluster_sum<5>(cl, &s_part[0][0], C, t5);
  if (tid == 0) {
    const double nb = sqrt(t5[0]);
    int go = 0;
    double rho = 0.0;
    if (!isfinite(nb)) {
      status = SLA_NONFINITE;
    } else if (nb == 0.0) {
      status = SLA_OK;
      pending = 2;
      if (rank == 0 && hist) hist[0] = 0.0;
    } else if (JAC && t5[3] > 0.0) {
      status = SLA_NONFINITE;
    } else if (JAC && t5[4] > 0.0) {
      status = SLA_BREAKDOWN;
    } else {
      const double rr = t5[1];
      rel = sqrt(rr) / nb;
      if (rank == 0 && hist) hist[0] = rel;
      if (!isfinite(rr)) status = SLA_NONFINITE;
      else if (sqrt(rr) <= P.rtol * nb) status = SLA_OK;
      else if (P.maxit == 0) status = SLA_NOT_CONVERGED;
      else {
        rho = JAC ? t5[2] : rr;
        go = 1;
      }
    }
    S.go = go;
    S.alpha = S.beta = S.alpha_prev = 0.0;
    s_vsc[0] = s_vsc[1] = s_vsc[2] = V(0);
    S.rho = rho;
    S.nb = nb;
    const double tol = P.rtol * nb, e4 = 4.0 * 2.220446049250313e-16;
    const double t1 = tol * (1.0 - e4), t2 = tol * (1.0 + e4);
    S.tol = tol;
    S.rr_lo = t1 * t1;
    S.rr_hi = t2 * t2;
  }
  __syncthreads();

  // ---- iterations
  SLA_PHASE_INIT();
  while (S.go) {
    const bool first = (k == 0);
    const V vb = s_vsc[0], va_prev = s_vsc[2];
    V *sp = (k & 1) ? sp1 : sp0;         // p_k (one buffer without two_p)
    const V *spo = (k & 1) ? sp0 : sp1;  // p_{k-1}
    // p_k (one buffer) or p_{k-1} (two_p) in a partner's layout
    const int64_t pp_off = (int64_t)cap * (two_p ? ((k & 1) ? 2 : 3) : 2);
    for (int li = tid; li < len; li += CB) {
      const V rl = sr[li];
      const V z = JAC ? sd[li] * rl : rl;
      V pv = z;
      if (!first) {
        const V po = spo[li];
        pv = fmav<V>(vb, po, z);
        sx[li] = fmav<V>(va_prev, po, sx[li]);
      }
      sp[li] = pv;
    }
    if (two_p) __syncthreads();  // this CTA's p_k is in place; the partners' is formed below
    else cl.sync();              // every CTA's p_k is in place
    SLA_PHASE(0);
    // p_k at column c: own rows from shared memory, a partner's through distributed shared memory
    auto p_at = [&](int32_t c) -> V {
      const uint32_t off = (uint32_t)((int64_t)c - c0);
      if (off < (uint32_t)len) return sp[off];
      if (!col_ok(c, (int32_t)n, &glob->bad_csr)) return V(0);
      // the partner owning c: a binary search over the partners' first rows (integer compares
      // only; C is a power of two <= 16)
      int j = 0;
#pragma unroll
      for (int step = kClMax / 2; step >= 1; step >>= 1)
        if (j + step < C && c >= s_start[j + step]) j += step;
      const V *px = s_peer[j];
      const int64_t o = (int64_t)c - s_start[j];
      if (!two_p) return px[pp_off + o];
      // the partner's own p_k expression from its r_k (1/diag) and p_{k-1}: the same bits
      const V rc = px[cap + o];
      const V zc = JAC ? px[sq_off + cap + o] * rc : rc;
      return first ? zc : fmav<V>(vb, px[pp_off + o], zc);
    };
    // Rows come in groups of kClGroup per thread: p.q is summed in the data type within a group
    // and the groups in fp64.  The group is an outer loop, so no fp64 instruction sits in the
    // per-row code (a predicated one would still occupy the fp64 unit on every row).
    V part = V(0);
    auto row_done = [&](int li, V acc) {
      sq[li] = acc;
      part = fmav<V>(sp[li], acc, part);
    };
    auto spmv_rows = [&](int gb, int ge) {
      if (rostaged && !mstaged) {
        // matrix streamed from L2/HBM: kClR rows per thread at a time, the first kClK entries of
        // each loaded together (independent loads in flight instead of one row's chain at a
        // time); every row still adds its entries in order
        const int32_t *__restrict__ cib = ci + m_lo;
        const V *__restrict__ vab = val + m_lo;
        for (int j0 = gb + tid; j0 < ge; j0 += kClR * CB) {
          int32_t eb[kClR], ee[kClR];
#pragma unroll
          for (int u = 0; u < kClR; ++u) {
            const int li = j0 + u * CB;
            eb[u] = li < ge ? s_ro[li] : 0;
            ee[u] = li < ge ? s_ro[li + 1] : 0;
          }
          int32_t cc[kClR][kClK];
          V vv[kClR][kClK];
#pragma unroll
          for (int t = 0; t < kClK; ++t)
#pragma unroll
            for (int u = 0; u < kClR; ++u) {
              const int32_t e = eb[u] + t;
              const bool in = e < ee[u];
              cc[u][t] = in ? __ldg(cib + e) : 0;
              vv[u][t] = in ? __ldg(vab + e) : V(0);
            }
          V acc[kClR];
#pragma unroll
          for (int u = 0; u < kClR; ++u) acc[u] = V(0);
#pragma unroll
          for (int t = 0; t < kClK; ++t)
#pragma unroll
            for (int u = 0; u < kClR; ++u)
              if (eb[u] + t < ee[u]) acc[u] = fmav<V>(vv[u][t], p_at(cc[u][t]), acc[u]);
#pragma unroll
          for (int u = 0; u < kClR; ++u)
            for (int32_t e = eb[u] + kClK; e < ee[u]; ++e)
              acc[u] = fmav<V>(__ldg(vab + e), p_at(__ldg(cib + e)), acc[u]);
#pragma unroll
          for (int u = 0; u < kClR; ++u) {
            const int li = j0 + u * CB;
            if (li < ge) row_done(li, acc[u]);
          }
        }
      } else {
        for (int li = gb + tid; li < ge; li += CB) {
          int64_t e0, e1;
          if (mstaged) {
            e0 = s_ro[li];
            e1 = s_ro[li + 1];
            if (e1 < e0) e1 = e0;
          } else {
            row_range(rp, c0 + li, P.nnz, e0, e1, &glob->bad_csr);
          }
          V acc = V(0);
          for (int64_t e = e0; e < e1; ++e) {
            const int32_t c = mstaged ? s_ci[e] : __ldg(ci + e);
            const V v = mstaged ? s_val[e] : __ldg(val + e);
            acc = fmav<V>(v, p_at(c), acc);
          }
          row_done(li, acc);
        }
      }
    };
    constexpr int kGrpRows = kClGroup * CB;
    spmv_rows(0, len < kGrpRows ? len : kGrpRows);
    double pqd = (double)part;
    for (int gb = kGrpRows; gb < len; gb += kGrpRows) {
      part = V(0);
      spmv_rows(gb, len - gb < kGrpRows ? len : gb + kGrpRows);
      pqd += (double)part;
    }
    SLA_PHASE(1);
    double v1[1] = {pqd};
    block_sum4<1, CB>(v1, s_red);
    if (tid == 0) s_part[1][0] = v1[0];
    cl.sync();
    double pqv[1];
    if (tid < 32) cluster_sum<1>(cl, &s_part[1][0], C, pqv);
    if (tid == 0) {
      const double pq = pqv[0];
      int go = 1;
      if (!isfinite(pq)) { status = SLA_NONFINITE; go = 0; }
      else if (!(pq > 0.0)) { status = SLA_BREAKDOWN; go = 0; }
      else {
        S.alpha = S.rho / pq;
        s_vsc[1] = (V)S.alpha;
      }
      S.go = go;
    }
    __syncthreads();
    SLA_PHASE(2);
    if (!S.go) break;
    const V va = s_vsc[1];
    double acc2[2] = {0.0, 0.0};
    V rr_t = V(0), rz_t = V(0);
    auto r_rows = [&](int gb, int ge) {
      for (int li = gb + tid; li < ge; li += CB) {
        const V ri = fmav<V>(-va, sq[li], sr[li]);
        sr[li] = ri;
        rr_t = fmav<V>(ri, ri, rr_t);
        if (JAC) rz_t = fmav<V>(ri, sd[li] * ri, rz_t);
      }
    };
    {
      constexpr int kGrpRows = kClGroup * CB;
      r_rows(0, len < kGrpRows ? len : kGrpRows);  // groups of rows as for p.q
      acc2[0] = (double)rr_t;
      if (JAC) acc2[1] = (double)rz_t;
      for (int gb = kGrpRows; gb < len; gb += kGrpRows) {
        rr_t = rz_t = V(0);
        r_rows(gb, len - gb < kGrpRows ? len : gb + kGrpRows);
        acc2[0] += (double)rr_t;
        if (JAC) acc2[1] += (double)rz_t;
      }
    }
    SLA_PHASE(3);
    if (JAC) {
      block_sum4<2, CB>(acc2, s_red);
    } else {
      double a1[1] = {acc2[0]};
      block_sum4<1, CB>(a1, s_red);
      acc2[0] = a1[0];
    }
    if (tid == 0) {
      s_part[0][0] = acc2[0];
      s_part[0][1] = acc2[1];
    }
    cl.sync();
    ++k;
    double t2[2] = {0.0, 0.0};
    if (tid < 32) {
      if (JAC) {
        cluster_sum<2>(cl, &s_part[0][0], C, t2);
      } else {
        double t1[1];
        cluster_sum<1>(cl, &s_part[0][0], C, t1);
        t2[0] = t1[0];
      }
    }
    if (tid == 0) {
      const double rrt = t2[0], rzt = t2[1];
      rr_last = rrt;
      if (rank == 0 && hist) hist[k] = rrt;  // turned into ||r|| / ||b|| after the loop
      int go = 0;
      pending = 1;
      if (!isfinite(rrt)) status = SLA_NONFINITE;
      else if (stop_test(rrt, S)) status = SLA_OK;
      else if (k >= P.maxit) status = SLA_NOT_CONVERGED;
      else {
        const double rho_new = JAC ? rzt : rrt;
        S.beta = rho_new / S.rho;
        S.rho = rho_new;
        S.alpha_prev = S.alpha;
        s_vsc[0] = (V)S.beta;
        s_vsc[2] = (V)S.alpha;
        pending = 0;
        go = 1;
      }
      S.go = go;
    }
    __syncthreads();
    SLA_PHASE(4);
  }
  SLA_PHASE_STORE(k);

  // ---- finish
  if (tid == 0) s_pending = pending;
  __syncthreads();
  const V va = (V)S.alpha;
  const V *sp_last = ((k - 1) & 1) ? sp1 : sp0;  // p of the last iteration
  for (int li = tid; li < len; li += CB) {
    V xv = sx[li];
    if (s_pending == 1) xv = fmav<V>(va, sp_last[li], xv);
    else if (s_pending == 2) xv = V(0);
    xg[c0 + li] = xv;
  }
  if (rank == 0 && hist && S.nb > 0.0) {
    const double nbs = S.nb;
    for (int64_t j = 1 + tid; j <= k; j += CB) hist[j] = sqrt(hist[j]) / nbs;
  }
  if (rank == 0 && tid == 0) {
    if (rr_last >= 0.0 || rr_last != rr_last) rel = sqrt(rr_last) / S.nb;
    Cs->k = k;
    Cs->status = status;
    Cs->rel_res = rel;
    Cs->nb = S.nb;
    Cs->alpha = S.alpha;
    Cs->beta = S.beta;
    Cs->rho = S.rho;
    Cs->done = 1;
  }
  cl.sync();  // no CTA leaves while a partner may still read its shared memory
}

}  // namespace

// Cluster shape for `batch` systems of n unknowns: C CTAs per system, rows per CTA (cap), threads
// per CTA, shared memory, and how many CSR entries a CTA may keep on chip (mcap, 0: none).  Every
// cluster runs a whole solve, so all of them must be resident at once: candidates are checked
// with the occupancy API and the first that fits in one wave is taken.
struct ClusterShape {
  int C = 0, cap = 0, block = 0, mcap = 0, ro = 0, two_p = 0;
  size_t smem = 0;
};

template <typename V, typename I, bool JAC>
ClusterShape cluster_shape_for(int64_t n, int64_t batch, int64_t nnz) {
  ClusterShape best;
  const ResidentLimits L = limits();
  if (n <= 0 || batch < 1 || L.sms <= 0 || batch > 65535) return best;
  const int nvec = JAC ? 5 : 4;
  static std::atomic<int> attr_set{0};
  if (!attr_set.load()) {
    for (void *f : {(void *)cg_cluster<V, I, JAC, 1024>, (void *)cg_cluster<V, I, JAC, 512>,
                    (void *)cg_cluster<V, I, JAC, kClBlock>}) {
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kClSmemMax) != cudaSuccess ||
          cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return best;
      }
    }
    attr_set.store(1);
  }
  int c0 = 1;
  while (c0 < kClMax && (int64_t)c0 * batch < L.sms) c0 *= 2;
  for (int c = c0; c <= kClMax; c *= 2) {
    if (c > n) break;
    const int64_t rows = (n + c - 1) / c;
    // on-chip staging of the CSR slice, decided with one p buffer: the slice on chip if it fits
    // beside the vectors (average row length plus slack), else the row offsets alone, so the
    // streamed SpMV starts from shared memory
    const int64_t ment = (nnz * rows) / std::max<int64_t>(n, 1) + 64;
    const size_t mat_bytes = (size_t)((rows + 1 + 3) & ~3) * 4 + (size_t)((ment + 3) & ~3) * 4 + (size_t)ment * sizeof(V);
    const size_t ro_bytes = (size_t)((rows + 1 + 3) & ~3) * 4;
    const size_t vec1 = (size_t)rows * nvec * sizeof(V);
    if (vec1 > kClSmemMax) continue;
    const bool keep_mat = vec1 + mat_bytes <= kClSmemMax;
    const bool keep_ro = SLA_CLUSTER_STAGE_RO && !keep_mat && vec1 + ro_bytes + 16 <= kClSmemMax;
    // block sizes in order of preference; for each, a second p buffer (one cluster barrier fewer
    // per iteration) when it fits with the same staging, else one
    for (int block : {rows >= 2048 ? 512 : kClBlock, kClBlock}) {
      for (int two_p = 1; two_p >= 0; --two_p) {
        const size_t vec_bytes = vec1 + (two_p ? (size_t)rows * sizeof(V) : 0);
        const size_t smem = vec_bytes + (keep_mat ? mat_bytes : 0) + (keep_ro ? ro_bytes : 0) + 16;
        if (smem > kClSmemMax) continue;
        void *fn = block == 512 ? (void *)cg_cluster<V, I, JAC, 512> : (void *)cg_cluster<V, I, JAC, kClBlock>;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)c;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(batch * c));
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, fn, &cfg) != cudaSuccess) {
          cudaGetLastError();
          continue;
        }
        if (active >= batch) {
          best.C = c;
          best.cap = (int)rows;
          best.block = block;
          best.mcap = keep_mat ? (int)ment : 0;
          best.ro = keep_ro ? 1 : 0;
          best.two_p = two_p;
          best.smem = smem;
          return best;
        }
      }
    }
  }
  return best;
}

template <typename V, typename I, bool JAC>
sla_status run_cluster(Prob<V, I> P, int64_t batch, cudaStream_t stream, sla_cg_info *info) {
  const ClusterShape sh = cluster_shape_for<V, I, JAC>(P.n, batch, P.nnz);
  if (sh.C == 0) return SLA_INVALID_ARG;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)sh.C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(batch * sh.C));
  cfg.blockDim = dim3(sh.block);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaMemsetAsync(P.glob, 0, sizeof(Glob), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(P.ctl, 0, sizeof(Ctl) * (size_t)batch, stream);
  if (e != cudaSuccess) return fail(e);
  if (sh.block == 512)
    e = cudaLaunchKernelEx(&cfg, cg_cluster<V, I, JAC, 512>, P, sh.C, sh.cap, sh.mcap, sh.ro, sh.two_p);
  else
    e = cudaLaunchKernelEx(&cfg, cg_cluster<V, I, JAC, kClBlock>, P, sh.C, sh.cap, sh.mcap, sh.ro, sh.two_p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  if (!info) return SLA_OK;
  return read_info(P.ctl, P.glob, batch, stream, info);
}

#define SLA_INSTANTIATE_CLUSTER(V, I, J) \
  template sla_status run_cluster<V, I, J>(Prob<V, I>, int64_t, cudaStream_t, sla_cg_info *);
SLA_INSTANTIATE_CLUSTER(double, int32_t, false)
SLA_INSTANTIATE_CLUSTER(double, int32_t, true)
SLA_INSTANTIATE_CLUSTER(double, int64_t, false)
SLA_INSTANTIATE_CLUSTER(double, int64_t, true)
SLA_INSTANTIATE_CLUSTER(float, int32_t, false)
SLA_INSTANTIATE_CLUSTER(float, int32_t, true)
SLA_INSTANTIATE_CLUSTER(float, int64_t, false)
SLA_INSTANTIATE_CLUSTER(float, int64_t, true)

bool cluster_fits(int64_t n, int64_t batch, int dtype, int precond) {
  // cheap necessary condition; run_cluster makes the final (occupancy) decision
  if (n <= 0 || batch < 1 || batch > 65535) return false;
  const int64_t rows = (n + kClMax - 1) / kClMax;
  const size_t vec_bytes = (size_t)rows * (precond == SLA_PRECOND_JACOBI ? 5 : 4) * (dtype == SLA_F64 ? 8 : 4);
  return vec_bytes <= kClSmemMax;
}

}  // namespace sla

#ifdef SLA_PHASE_TIMING
extern "C" SLA_API int sla_cluster_phase_cycles(unsigned long long *host, int nblocks) {
  return (int)cudaMemcpyFromSymbol(host, sla::g_phase_cycles, sizeof(unsigned long long) * 8 * (size_t)nblocks);
}
#endif
