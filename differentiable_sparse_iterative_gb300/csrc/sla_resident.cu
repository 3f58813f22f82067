// Resident CG: the whole solve in one persistent kernel, vectors kept in shared memory.
//
// Method as in sla_cg.cu ("torch-sla" technical summary, Methodology 1-2 and Significance:
// Hestenes-Stiefel CG with optional Jacobi preconditioning; same recurrences, same stopping
// rule, same status decisions).
//
// GB300 design.  When one system fits on chip (r, p and, with Jacobi, 1/diag for a 1/G
// share of the rows in one SM's 227 KB of shared memory), one 1024-thread block per SM owns
// a contiguous row chunk for the whole solve; r and p never leave the SM, while x and q,
// each touched once per iteration, live in global memory and stay in L2.  Per iteration the
// matrix is streamed (from L2 when it fits there) and the values the neighbouring blocks
// need are published: r_k and p_{k-1}, from which a block recomputes p_k = z + beta p_{k-1}
// for the few columns outside its chunk.  The two global dependencies
// of an iteration (alpha needs p.Ap, beta needs r.r) are two grid barriers, each carrying
// a deterministic all-reduce: every block writes its block sum, and after the barrier every
// block adds the G block sums in the same fixed order, so all blocks hold bit-identical
// scalars and take the same branch.  The launch is cooperative (all blocks co-resident);
// each barrier wait is bounded and ends the solve with SLA_TIMEOUT if it ever expires.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "sla_common.cuh"
#include "sla_host.h"
#include "sla_grid.cuh"
#include "sla_onchip.cuh"

namespace sla {

namespace {

constexpr int kResBlock = 1024;
static_assert(kResBlock == kPublishBlock, "block sums go through block_publish");
constexpr int kStage = 8;  // rows per thread whose global loads are issued together
constexpr long long kSpinLimit = 1ll << 26;  // ~seconds of polling before a barrier gives up

// Grid-barrier wait bounds of the next launches (sla_test_set_barrier_wait; normally 0 and kSpinLimit).
std::atomic<unsigned> g_wait_extra{0u};
std::atomic<long long> g_wait_limit{kSpinLimit};

// p_k at a column outside the block's chunk, from the published r_k and p_{k-1}.
template <typename V, bool JAC>
__device__ __forceinline__ V p_remote(const V *r, const V *dinv, const V *po, int32_t c, bool first, V beta) {
  const V rc = __ldcg(r + c);
  const V zc = JAC ? __ldcg(dinv + c) * rc : rc;
  return first ? zc : fmav<V>(beta, __ldcg(po + c), zc);
}

template <typename V, typename I, bool JAC>
__global__ void __launch_bounds__(kResBlock, 1) cg_resident(Prob<V, I> P, int cap, WaitCfg wc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // shared: reduction buffer (2 x kResBlock doubles), then r, p (and 1/diag) of the block's rows
  double *sbuf = reinterpret_cast<double *>(smem_raw);
  V *sr = reinterpret_cast<V *>(sbuf + 2 * kResBlock);
  V *sp = sr + cap;
  V *sd = JAC ? sp + cap : nullptr;
  // halo bits of the block's rows (bit i: row i is read by another block), words from c0 / 32
  uint32_t *s_halo = reinterpret_cast<uint32_t *>((JAC ? sd : sp) + cap);
  __shared__ ResScalars S;
  const unsigned G = gridDim.x;
  const int bid = blockIdx.x, tid = threadIdx.x;
  const int64_t c0 = (int64_t)P.n * bid / G, c1 = (int64_t)P.n * (bid + 1) / G;
  const int len = (int)(c1 - c0);
  Glob *glob = P.glob;
  Ctl *C = P.ctl;
  unsigned *arrive = &glob->barrier;  // zeroed before the launch
  unsigned *timeout = &glob->timeout;
  // Partial-sum rows: 0..4 for the setup sums and later r.r, r.z (a block writes those only after
  // the p.q barrier, when every block has read the setup sums); row 5 for p.q.
  static_assert(kRedSlots >= 6, "the resident kernel needs 6 partial-sum rows");
  double *partB = P.partials;
  double *partA = P.partials + (size_t)5 * kMaxBlocksPerSystem;
  const I *__restrict__ rp = P.rp;
  const int32_t *__restrict__ ci = P.ci;
  const V *__restrict__ val = P.val;
  V *rpub = P.r;        // published r_k (read by the neighbouring blocks)
  V *dpub = P.dinv;     // published 1/diag (Jacobi)
  V *xg = P.x;          // x stays in global memory (L2): read and written once per iteration
  V *qg = P.q;          // q likewise, between the SpMV and the r update
  unsigned epoch = 0;
  if (bid == 0 && tid == 0) atomicAdd(&glob->kernels, 1ull);

  // ---- setup: x = x0 (or 0), r = b - A x0, 1/diag; sums b.b, r.r, r.z, #non-finite, #non-positive
  double acc5[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
  for (int li = tid; li < len; li += kResBlock) {
    const int64_t i = c0 + li;
    int64_t e0, e1;
    row_range(rp, i, P.nnz, e0, e1, &glob->bad_csr);
    const V bi = P.b[i];
    V ri = bi;
    if (P.x0) {
      V s_ = V(0);
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = ci[e];
        if (col_ok(c, P.n, &glob->bad_csr)) s_ = fmav<V>(val[e], P.x0[c], s_);
      }
      ri = bi - s_;
    }
    sr[li] = ri;
    rpub[i] = ri;
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
      dpub[i] = di;
      acc5[2] = fma((double)ri, (double)(di * ri), acc5[2]);
    }
  }
  // Mark the rows this block reads from other blocks.  Each iteration a block then publishes r
  // and p for its marked rows only (for a grid stencil about 30 % of them); the others never
  // leave shared memory.  Without the bitmap (P.halo NULL) every row is published.
  const bool has_halo = P.halo != nullptr;
  if (has_halo) {
    for (int li = tid; li < len; li += kResBlock) {
      int64_t e0, e1;
      row_range(rp, c0 + li, P.nnz, e0, e1, &glob->bad_csr);
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = ci[e];
        if ((uint32_t)c < (uint32_t)P.n && ((int64_t)c < c0 || (int64_t)c >= c1))
          atomicOr(P.halo + (c >> 5), 1u << (c & 31));
      }
    }
  }
  // x = x0 (or 0) after every block has read x0 (x0 may be the same buffer as x)
  block_publish<5>(acc5, sbuf, partB);
  const bool ok0 = grid_barrier(arrive, timeout, G, epoch, wc);
  for (int li = tid; li < len; li += kResBlock) xg[c0 + li] = P.x0 ? P.x0[c0 + li] : V(0);
  const int64_t hw0 = c0 >> 5;  // first bitmap word of the block's rows
  if (has_halo && len > 0)
    for (int64_t w = hw0 + tid; w <= ((c1 - 1) >> 5); w += kResBlock) s_halo[w - hw0] = __ldcg(P.halo + w);
  auto published = [&](int li) -> bool {
    const int64_t i = c0 + li;
    return !has_halo || ((s_halo[(i >> 5) - hw0] >> (i & 31)) & 1u);
  };

  // thread 0 of every block takes the same decisions from the same totals
  int status = SLA_NOT_CONVERGED, pending = 0;
  int64_t k = 0;
  double nb = 0.0, rel = 0.0, rho = 0.0, rr_last = -1.0;
  if (tid < 32) {
    double t5[5];
    warp_totals<5>(partB, (int)G, t5);
    if (tid == 0) {
      nb = sqrt(t5[0]);
      int go = 0;
      if (!ok0) {
        status = SLA_TIMEOUT;
      } else if (!isfinite(nb)) {
        status = SLA_NONFINITE;
      } else if (nb == 0.0) {
        status = SLA_OK;
        pending = 2;
        if (bid == 0 && P.history) P.history[0] = 0.0;
      } else if (JAC && t5[3] > 0.0) {
        status = SLA_NONFINITE;
      } else if (JAC && t5[4] > 0.0) {
        status = SLA_BREAKDOWN;
      } else {
        const double rr = t5[1];
        rel = sqrt(rr) / nb;
        if (bid == 0 && P.history) P.history[0] = rel;
        if (!isfinite(rr)) status = SLA_NONFINITE;
        else if (sqrt(rr) <= P.rtol * nb) status = SLA_OK;
        else if (P.maxit == 0) status = SLA_NOT_CONVERGED;
        else {
          rho = JAC ? t5[2] : rr;
          go = 1;
        }
      }
      S.go = go;
      S.alpha = 0.0;
      S.beta = 0.0;
      S.alpha_prev = 0.0;
      S.rho = rho;
      S.nb = nb;
      const double tol = P.rtol * nb, e4 = 4.0 * 2.220446049250313e-16;
      const double t1 = tol * (1.0 - e4), t2 = tol * (1.0 + e4);
      S.tol = tol;
      S.rr_lo = t1 * t1;
      S.rr_hi = t2 * t2;
    }
  }
  __syncthreads();

  // ---- iterations
  SLA_PHASE_INIT();
  while (S.go) {
    const int par = (int)(k & 1);
    const bool first = (k == 0);
    const V vb = (V)S.beta;
    V *pn_pub = P.p[par];
    const V *po_pub = P.p[par ^ 1];
    // p_k = z_k + beta p_{k-1} for the own rows; publish p_k
    for (int li = tid; li < len; li += kResBlock) {
      const V rl = sr[li];
      const V z = JAC ? sd[li] * rl : rl;
      const V pv = first ? z : fmav<V>(vb, sp[li], z);
      sp[li] = pv;
      if (published(li)) pn_pub[c0 + li] = pv;
    }
    __syncthreads();
    SLA_PHASE(0);
    // q = A p_k and the block's share of p.q (row pointers of a group loaded up front)
    V part = V(0);
    for (int j0 = tid; j0 < len; j0 += kStage * kResBlock) {
      I rpa[kStage], rpb[kStage];
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
        const int li = j0 + u * kResBlock;
        rpa[u] = li < len ? __ldg(rp + c0 + li) : I(0);
        rpb[u] = li < len ? __ldg(rp + c0 + li + 1) : I(0);
      }
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
      const int li = j0 + u * kResBlock;
      // warps with no row left branch around (fp64 instructions issued with every lane
      // predicated off would still occupy the fp64 unit); lanes past the outer loop's end are
      // not active, hence the active mask
      if (!__any_sync(__activemask(), li < len)) break;
      if (li >= len) continue;
      const int64_t i = c0 + li;
      int64_t e0 = (int64_t)rpa[u], e1 = (int64_t)rpb[u];
      if (e0 < 0 || e1 < e0 || e1 > P.nnz) {
        atomicOr(&glob->bad_csr, 1u);
        e0 = e1 = 0;
      }
      V acc = V(0);
      for (int64_t e = e0; e < e1; ++e) {
        const int32_t c = __ldg(ci + e);
        const V v = __ldg(val + e);
        const uint32_t off = (uint32_t)((int64_t)c - c0);
        V pc;
        if (off < (uint32_t)len) pc = sp[off];
        else pc = col_ok(c, P.n, &glob->bad_csr) ? p_remote<V, JAC>(rpub, dpub, po_pub, c, first, vb) : V(0);
        acc = fmav<V>(v, pc, acc);
      }
      qg[i] = acc;
      part = fmav<V>(sp[li], acc, part);
      }
    }
    const double v1[1] = {(double)part};
    SLA_PHASE(1);
    block_publish<1>(v1, sbuf, partA);
    const bool ok1 = grid_barrier(arrive, timeout, G, epoch, wc);
    SLA_PHASE(2);
    if (tid < 32) {
      double t1[1];
      warp_totals<1>(partA, (int)G, t1);
      if (tid == 0) {
        const double pq = t1[0];
        int go = 1;
        if (!ok1) { status = SLA_TIMEOUT; go = 0; }
        else if (!isfinite(pq)) { status = SLA_NONFINITE; go = 0; }
        else if (!(pq > 0.0)) { status = SLA_BREAKDOWN; go = 0; }
        else S.alpha = rho / pq;
        S.go = go;
      }
    }
    __syncthreads();
    if (!S.go) break;
    // r -= alpha q; publish r; sums r.r (and r.z).  float data: each group of kStage rows is
    // summed in float, then added to the fp64 sums.
    const V va = (V)S.alpha;
    double acc2[2] = {0.0, 0.0};
    // fp64 data: one FMA chain over all of the thread's rows (no extra fp64 adds); fp32 data: a
    // float sum per stage, the stages added in fp64
    V rr_t = V(0), rz_t = V(0);
    bool flushed = false;
    for (int j0 = tid; j0 < len; j0 += kStage * kResBlock) {
      V qv[kStage];
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
        const int li = j0 + u * kResBlock;
        qv[u] = li < len ? qg[c0 + li] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
        const int li = j0 + u * kResBlock;
        if (!__any_sync(__activemask(), li < len)) break;  // as in the SpMV
        if (li < len) {
          const V ri = fmav<V>(-va, qv[u], sr[li]);
          sr[li] = ri;
          if (published(li)) rpub[c0 + li] = ri;
          rr_t = fmav<V>(ri, ri, rr_t);
          if (JAC) rz_t = fmav<V>(ri, sd[li] * ri, rz_t);
        }
      }
      if constexpr (sizeof(V) == 4) {
        acc2[0] = flushed ? acc2[0] + (double)rr_t : (double)rr_t;
        if (JAC) acc2[1] = flushed ? acc2[1] + (double)rz_t : (double)rz_t;
        flushed = true;
        rr_t = rz_t = V(0);
      }
    }
    if constexpr (sizeof(V) == 8) {
      acc2[0] = rr_t;
      if (JAC) acc2[1] = rz_t;
    }
    SLA_PHASE(3);
    if (JAC) {
      block_publish<2>(acc2, sbuf, partB);
    } else {
      const double v1r[1] = {acc2[0]};
      block_publish<1>(v1r, sbuf, partB);
    }
    grid_arrive(arrive, epoch);
    // while the other blocks arrive: x_{k+1} = x_k + alpha_k p_k, which needs neither reduction
    // (p_k is still in shared memory); whatever the r.r test decides, this update is due
    for (int j0 = tid; j0 < len; j0 += kStage * kResBlock) {
      V xv[kStage];
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
        const int li = j0 + u * kResBlock;
        xv[u] = li < len ? xg[c0 + li] : V(0);
      }
#pragma unroll
      for (int u = 0; u < kStage; ++u) {
        const int li = j0 + u * kResBlock;
        if (!__any_sync(__activemask(), li < len)) break;  // as in the SpMV
        if (li < len) xg[c0 + li] = fmav<V>(va, sp[li], xv[u]);
      }
    }
    const bool ok2 = grid_wait(arrive, timeout, G, epoch, wc);
    SLA_PHASE(4);
    ++k;
    if (tid < 32) {
      double t2[2] = {0.0, 0.0};
      if (JAC) warp_totals<2>(partB, (int)G, t2);
      else {
        double t1[1];
        warp_totals<1>(partB, (int)G, t1);
        t2[0] = t1[0];
      }
      // lane 0 the stopping test, lane 1 beta (in parallel); the history keeps r.r for now and is
      // turned into ||r|| / ||b|| after the loop
      const double rrt = t2[0];
      const double rho_new = JAC ? t2[1] : rrt;
      double lane_val = 0.0;
      if (tid == 1) lane_val = rho_new / S.rho;
      if (tid == 2 && bid == 0 && P.history) P.history[k] = rrt;
      int stop_code = 0;  // 0 go on, 1 converged, 2 non-finite, 3 maxit, 4 timeout
      if (tid == 0) {
        if (!ok2) stop_code = 4;
        else if (!isfinite(rrt)) stop_code = 2;
        else if (stop_test(rrt, S)) stop_code = 1;
        else if (k >= P.maxit) stop_code = 3;
      }
      const double beta_new = __shfl_sync(0xffffffffu, lane_val, 1);
      if (tid == 0) {
        rr_last = rrt;
        int go = 0;
        if (stop_code == 4) status = SLA_TIMEOUT;
        else if (stop_code == 2) status = SLA_NONFINITE;
        else if (stop_code == 1) status = SLA_OK;
        else if (stop_code == 3) status = SLA_NOT_CONVERGED;
        else {
          S.beta = beta_new;
          S.rho = rho_new;
          rho = rho_new;
          S.alpha_prev = S.alpha;
          go = 1;
        }
        S.go = go;
      }
    }
    __syncthreads();
    SLA_PHASE(5);
  }
  SLA_PHASE_STORE(k);

  // ---- finish: x = 0 for b = 0 (every other x update was made inside the loop)
  __shared__ int s_pending;
  if (tid == 0) s_pending = pending;
  __syncthreads();
  if (s_pending == 2) {
    for (int li = tid; li < len; li += kResBlock) xg[c0 + li] = V(0);
  }
  // history entries 1..k hold r.r: convert them to ||r|| / ||b|| (block 0, all threads)
  if (bid == 0 && P.history && S.nb > 0.0) {
    const double nbs = S.nb;
    for (int64_t j = 1 + tid; j <= k; j += kResBlock) P.history[j] = sqrt(P.history[j]) / nbs;
  }
  if (bid == 0 && tid == 0) {
    if (rr_last >= 0.0 || rr_last != rr_last) rel = sqrt(rr_last) / nb;
    C->k = k;
    C->status = status;
    C->rel_res = rel;
    C->nb = nb;
    C->alpha = S.alpha;
    C->beta = S.beta;
    C->rho = rho;
    C->done = 1;
  }
}

constexpr size_t kResStaticSmem = 4096;  // reduction scratch and flags of the kernel itself


// Blocks and rows per block for the resident kernel, or G = 0 if the system does not fit.
void resident_shape(int64_t n, size_t vbytes, bool jac, const ResidentLimits &L, int64_t maxit, int &G,
                    int &cap, size_t &smem) {
  G = 0;
  cap = 0;
  smem = 0;
  if (n <= 0 || L.sms <= 0) return;
  const int nvec = jac ? 3 : 2;  // r, p (and 1/diag) stay in shared memory; x and q live in L2
  int g = (int)std::min<int64_t>(L.sms, std::max<int64_t>(1, (n + 255) / 256));
  g = std::min(g, kMaxBlocksPerSystem);
  const int64_t rows = (n + g - 1) / g;
  // reduction buffer, r, p (1/diag) of the rows, and their halo bitmap words (rows / 32 + 2)
  const size_t need = (size_t)2 * kResBlock * sizeof(double) + (size_t)rows * nvec * vbytes +
                      sizeof(uint32_t) * (size_t)(rows / 32 + 2);
  if (need + kResStaticSmem > (size_t)L.max_smem) return;
  // the barrier counter counts 2 barriers per iteration plus setup, G arrivals each
  if ((double)(2 * maxit + 2) * g >= 4.0e9) return;
  G = g;
  cap = (int)rows;
  smem = need;
}

}  // namespace

bool resident_fits(int64_t n, int64_t batch, int dtype, int precond, int64_t maxit) {
  if (batch != 1) return false;
  int G, cap;
  size_t smem;
  resident_shape(n, dtype == SLA_F64 ? 8 : 4, precond == SLA_PRECOND_JACOBI, limits(), maxit, G, cap, smem);
  return G > 0;
}

template <typename V, typename I, bool JAC>
sla_status run_resident(Prob<V, I> P, cudaStream_t stream, sla_cg_info *info) {
  int G, cap;
  size_t smem;
  if (P.batch != 1) return SLA_INVALID_ARG;  // one system per resident launch
  resident_shape(P.n, sizeof(V), JAC, limits(), P.maxit, G, cap, smem);
  if (G == 0) return SLA_INVALID_ARG;
  P.G = G;
  void *fn = (void *)cg_resident<V, I, JAC>;
  static std::atomic<size_t> smem_set{0};
  if (smem_set.load() < smem) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(e);
    smem_set.store(smem);
  }
  // fresh loop state: counters, flags and the control block start at zero
  cudaError_t e = cudaMemsetAsync(P.glob, 0, sizeof(Glob), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(P.ctl, 0, sizeof(Ctl), stream);
  if (e == cudaSuccess && P.halo)
    e = cudaMemsetAsync(P.halo, 0, sizeof(uint32_t) * (size_t)((P.n + 31) / 32), stream);
  if (e != cudaSuccess) return fail(e);
  WaitCfg wc = launch_wait_cfg();
  void *args[] = {(void *)&P, (void *)&cap, (void *)&wc};
  e = cudaLaunchCooperativeKernel(fn, dim3(G), dim3(kResBlock), args, smem, stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    // not every block can be resident at once here (e.g. a GPU shared by SM partitioning): the
    // launch is refused before anything runs and the context is unaffected; SLA_INVALID_ARG lets
    // the automatic engine choice move on to the graph loop
    cudaGetLastError();
    return SLA_INVALID_ARG;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  if (!info) return SLA_OK;
  sla_status s = read_info(P.ctl, P.glob, 1, stream, info);
  return s;
}

#define SLA_INSTANTIATE_RESIDENT(V, I, J) \
  template sla_status run_resident<V, I, J>(Prob<V, I>, cudaStream_t, sla_cg_info *);
SLA_INSTANTIATE_RESIDENT(double, int32_t, false)
SLA_INSTANTIATE_RESIDENT(double, int32_t, true)
SLA_INSTANTIATE_RESIDENT(double, int64_t, false)
SLA_INSTANTIATE_RESIDENT(double, int64_t, true)
SLA_INSTANTIATE_RESIDENT(float, int32_t, false)
SLA_INSTANTIATE_RESIDENT(float, int32_t, true)
SLA_INSTANTIATE_RESIDENT(float, int64_t, false)
SLA_INSTANTIATE_RESIDENT(float, int64_t, true)

}  // namespace sla

#ifdef SLA_PHASE_TIMING
extern "C" SLA_API int sla_phase_cycles(unsigned long long *host, int nblocks) {
  return (int)cudaMemcpyFromSymbol(host, sla::g_phase_cycles, sizeof(unsigned long long) * 8 * (size_t)nblocks);
}
#endif

namespace sla {
WaitCfg launch_wait_cfg() { return WaitCfg{g_wait_extra.load(), g_wait_limit.load()}; }
}  // namespace sla

extern "C" sla_status sla_test_set_barrier_wait(uint32_t extra, int64_t spin_limit) {
  if (extra > 1u || spin_limit < 0 || spin_limit > sla::kSpinLimit) return SLA_INVALID_ARG;
  sla::g_wait_extra.store(extra);
  sla::g_wait_limit.store(spin_limit == 0 ? sla::kSpinLimit : spin_limit);
  return SLA_OK;
}
