// Conjugate-gradient solve and adjoint backward on the GPU (libsla).
//
// Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers
// and Sparse Tensor Parallelism for PyTorch" (Chi, Wen), technical summary:
//   Methodology 1 - the GPU iterative backend (CG) behind .solve, one matrix
//     or a batch sharing one pattern;
//   Methodology 2 - linear-system adjoint: A^T lambda = dL/dx, grad_b = lambda,
//     grad_A = -lambda_i x_j on the pattern, O(n + nnz) memory;
//   Significance - Jacobi preconditioning of the native backend.
// Hestenes-Stiefel CG with the stopping rule ||r_k|| <= rtol ||b|| on the
// recursive residual (textbook reading; the summary gives no variant).
//
// GB300 design.  fp64 FMA issues at about 2 per clock per SM on this part, so
// one fp64 operation costs as much time as ~11 bytes of HBM traffic; each
// iteration is two fused kernels that keep the fp64 work near its minimum
// (about 10 operations per row for a five-point matrix) while streaming the
// matrix once:
//   K_A (spmv_step):   p_k = z_k + beta p_{k-1} for the block's rows (kept in
//                      shared memory), x += alpha_{k-1} p_{k-1} (delayed by one
//                      iteration so p_{k-1} is read once), q = A p_k with
//                      neighbours outside the tile recomputed from r and
//                      p_{k-1}, and the partial sums of p.q;
//   K_B (update_step): r -= alpha q and the partial sums of r.r (and r.z).
// Each kernel ends with a deterministic two-level reduction: every block
// publishes its partial sum, the last block to arrive adds all partials in a
// fixed order and computes alpha (K_A) or beta and the stopping test (K_B) on
// the device.  The loop itself is a CUDA graph: an init and a setup kernel,
// then a device-side conditional WHILE node whose body holds U iterations and a
// one-thread control kernel that ends the loop when every system has stopped,
// then a finish kernel that applies the last delayed x update.  The host
// launches one graph per solve and synchronises once to read the status.
// The kernels are in sla_stream.cuh; this file holds the host side (graph
// loop, host loop, engine choice) and the C entry points.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "sla_common.cuh"
#include "sla_host.h"
#include "sla_stream.cuh"
#include "sla_tma.cuh"

namespace sla {

// ------------------------------------------------------------------------ host side

namespace {

constexpr int kRPT = SLA_SPMV_RPT;
constexpr int kDefaultUnroll = 8;

// A cached graph loop.  Its key is the graph's shape (types, launch shape, unroll, device); the
// buffers and scalars of a call are kernel arguments, so a call of the same shape with other
// buffers reuses the instantiated graph after its nodes' arguments are replaced (`nodes` in the
// order of graph_node_params; `args` the problem they were last set for).
struct GraphEntry {
  std::vector<char> key;
  std::vector<char> args;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphConditionalHandle handle = 0;
  std::vector<cudaGraphNode_t> nodes;
  uint64_t stamp = 0;
};

std::mutex g_mu;
std::vector<GraphEntry> g_cache;
uint64_t g_stamp = 0;
uint64_t g_builds = 0, g_updates = 0;  // graphs instantiated; cached graphs pointed at a new problem
constexpr size_t kCacheCap = 32;

template <typename V, typename I, bool JAC>
struct Kernels {
  static void *init() { return (void *)cg_init<V, I>; }
  static void *setup() { return (void *)cg_setup<V, I, JAC>; }
  static void *spmv_step() { return (void *)cg_spmv_step<V, I, JAC, kRPT>; }
  static void *spmv_step_tma() { return (void *)cg_spmv_step_tma<V, I, JAC>; }
  static void *update_step() { return (void *)cg_update_step<V, I, JAC>; }
  static void *finish() { return (void *)cg_finish<V, I>; }
};

// Launch shape of the streaming path: blocks per system for the SpMV step and for the other
// kernels, and whether the SpMV step is the TMA-staged one (with its dynamic shared memory).
struct Launch {
  int G_main = 1;
  int G_spmv = 1;
  bool tma = false;
  unsigned tma_smem = 0;
};

// Arguments of the graph loop's kernel nodes for one problem (the arrays point into this object,
// which therefore stays where it was built).  Nodes, in order: init, setup, then per unrolled
// iteration u the SpMV step and the update step (parity u & 1), the loop control, finish.
template <typename V, typename I>
struct GraphArgs {
  Prob<V, I> P, Ps;
  int par[2] = {0, 1};
  Glob *gp;
  cudaGraphConditionalHandle h;
  uint32_t max_bodies;
  void *args_p[1];
  void *args_pp[2][2];
  void *args_ps[2][2];
  void *args_c[3];
  GraphArgs(const Prob<V, I> &P0, const Launch &Lc, int unroll, cudaGraphConditionalHandle h_) : P(P0), Ps(P0) {
    P.G = Lc.G_main;
    Ps.G = Lc.G_spmv;
    gp = P.glob;
    h = h_;
    max_bodies = (uint32_t)std::min<int64_t>((P.maxit + unroll - 1) / unroll + 2, 0x7fffffff);
    args_p[0] = &P;
    for (int q = 0; q < 2; ++q) {
      args_pp[q][0] = &P;
      args_pp[q][1] = &par[q];
      args_ps[q][0] = &Ps;
      args_ps[q][1] = &par[q];
    }
    args_c[0] = &gp;
    args_c[1] = &h;
    args_c[2] = &max_bodies;
  }
  GraphArgs(const GraphArgs &) = delete;
  GraphArgs &operator=(const GraphArgs &) = delete;
};

template <typename V, typename I, bool JAC>
cudaKernelNodeParams graph_node_params(GraphArgs<V, I> &A, const Launch &Lc, int unroll, int idx) {
  using K = Kernels<V, I, JAC>;
  cudaKernelNodeParams kp;
  memset(&kp, 0, sizeof(kp));
  const dim3 grid(A.P.G, A.P.batch), block(kBlock);
  const int nbody = 2 * unroll;
  if (idx == 0) {
    kp.func = K::init();
    kp.gridDim = dim3(1);
    kp.blockDim = block;
    kp.kernelParams = A.args_p;
  } else if (idx == 1) {
    kp.func = K::setup();
    kp.gridDim = grid;
    kp.blockDim = block;
    kp.kernelParams = A.args_p;
  } else if (idx < 2 + nbody) {
    const int u = (idx - 2) / 2;
    if (((idx - 2) & 1) == 0) {
      kp.func = Lc.tma ? K::spmv_step_tma() : K::spmv_step();
      kp.gridDim = dim3(A.Ps.G, A.P.batch);
      kp.blockDim = dim3(Lc.tma ? kTmaBlock : kBlock);
      kp.sharedMemBytes = Lc.tma ? Lc.tma_smem : 0u;
      kp.kernelParams = A.args_ps[u & 1];
    } else {
      kp.func = K::update_step();
      kp.gridDim = grid;
      kp.blockDim = block;
      kp.kernelParams = A.args_pp[u & 1];
    }
  } else if (idx == 2 + nbody) {
    kp.func = (void *)cg_loop_control;
    kp.gridDim = dim3(1);
    kp.blockDim = dim3(32);
    kp.kernelParams = A.args_c;
  } else {
    kp.func = K::finish();
    kp.gridDim = grid;
    kp.blockDim = block;
    kp.kernelParams = A.args_p;
  }
  return kp;
}

// The graph loop: init, setup, a conditional WHILE node whose body runs `unroll` iterations and
// the loop control, then finish.
template <typename V, typename I, bool JAC>
cudaError_t build_graph(const Prob<V, I> &P0, const Launch &Lc, int unroll, GraphEntry &en) {
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaGraphCreate(&g, 0);
  if (e != cudaSuccess) return e;
  cudaGraphConditionalHandle h;
  const int nbody = 2 * unroll;
  std::vector<cudaGraphNode_t> nodes((size_t)nbody + 4);
  cudaGraphNodeParams cp = {cudaGraphNodeTypeConditional};
  do {
    if ((e = cudaGraphConditionalHandleCreate(&h, g, 1u, cudaGraphCondAssignDefault)) != cudaSuccess) break;
    GraphArgs<V, I> A(P0, Lc, unroll, h);
    auto add = [&](int idx, cudaGraph_t gr, const cudaGraphNode_t *dep) {
      const cudaKernelNodeParams kp = graph_node_params<V, I, JAC>(A, Lc, unroll, idx);
      return cudaGraphAddKernelNode(&nodes[(size_t)idx], gr, dep, dep ? 1 : 0, &kp);
    };
    if ((e = add(0, g, nullptr)) != cudaSuccess) break;
    if ((e = add(1, g, &nodes[0])) != cudaSuccess) break;
    cudaGraphNode_t n_while;
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = h;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    if ((e = cudaGraphAddNode(&n_while, g, &nodes[1], nullptr, 1, &cp)) != cudaSuccess) break;
    cudaGraph_t body = cp.conditional.phGraph_out[0];
    for (int idx = 2; idx <= 2 + nbody && e == cudaSuccess; ++idx)
      e = add(idx, body, idx > 2 ? &nodes[(size_t)idx - 1] : nullptr);
    if (e != cudaSuccess) break;
    if ((e = add(3 + nbody, g, &n_while)) != cudaSuccess) break;
    e = cudaGraphInstantiate(&en.exec, g, 0);
  } while (0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return e;
  }
  en.graph = g;
  en.handle = h;
  en.nodes = std::move(nodes);
  return cudaSuccess;
}

// Points the nodes of a cached graph at another problem of the same shape (later launches only).
template <typename V, typename I, bool JAC>
cudaError_t update_graph(const Prob<V, I> &P0, const Launch &Lc, int unroll, GraphEntry &en) {
  GraphArgs<V, I> A(P0, Lc, unroll, en.handle);
  for (size_t idx = 0; idx < en.nodes.size(); ++idx) {
    const cudaKernelNodeParams kp = graph_node_params<V, I, JAC>(A, Lc, unroll, (int)idx);
    const cudaError_t e = cudaGraphExecKernelNodeSetParams(en.exec, en.nodes[idx], &kp);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The TMA-staged SpMV step is opt-in (sla_set_spmv_variant): measured on GB300 it is slower than
// the plain step on the five-point workloads (its per-entry staging bookkeeping makes it
// instruction-bound), so the plain step is the default.  Both compute the same rows.
std::atomic<int> g_spmv_variant{SLA_SPMV_PLAIN};

bool tma_enabled() { return g_spmv_variant.load() == SLA_SPMV_TMA; }

int occupancy_blocks(const void *fn) {
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kBlock, 0) != cudaSuccess || nb < 1) nb = 1;
  return nb;
}

struct DeviceInfo {
  int dev = -1;
  int sms = 0;
};

DeviceInfo device_info() {
  DeviceInfo d;
  cudaGetDevice(&d.dev);
  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, d.dev);
  if (d.sms < 1) d.sms = 1;
  return d;
}

// Blocks per system: fill the GPU once (SMs x resident blocks), at least 256 rows per block.
int choose_G(int64_t n, int64_t batch, int sms, int occ) {
  int64_t total = (int64_t)sms * occ;
  int64_t g = std::max<int64_t>(1, total / std::max<int64_t>(1, batch));
  g = std::min<int64_t>(g, (n + kBlock - 1) / kBlock);
  g = std::min<int64_t>(g, kMaxBlocksPerSystem);
  return (int)std::max<int64_t>(1, g);
}

// Host-driven loop: the same kernels launched directly; the host reads the number of active
// systems every `unroll` iterations (one 4-byte copy and one stream synchronisation).
template <typename V, typename I, bool JAC>
sla_status run_cg_host_loop(Prob<V, I> P, const Launch &Lc, int unroll, cudaStream_t stream, sla_cg_info *info,
                            int64_t batch) {
  P.G = Lc.G_main;
  Prob<V, I> Ps = P;
  Ps.G = Lc.G_spmv;
  dim3 grid(P.G, P.batch), grid_s(Ps.G, P.batch), block(kBlock);
  uint64_t launched = 0;
  cg_init<V, I><<<1, block, 0, stream>>>(P);
  cg_setup<V, I, JAC><<<grid, block, 0, stream>>>(P);
  launched += 2;
  uint32_t active = 1;
  for (int64_t k = 0; k < P.maxit && active; k += unroll) {
    const int64_t upto = std::min<int64_t>(P.maxit - k, unroll);
    for (int64_t u = 0; u < upto; ++u) {
      const int par = (int)((k + u) & 1);
      if (Lc.tma)
        cg_spmv_step_tma<V, I, JAC><<<grid_s, dim3(kTmaBlock), Lc.tma_smem, stream>>>(Ps, par);
      else
        cg_spmv_step<V, I, JAC, kRPT><<<grid_s, block, 0, stream>>>(Ps, par);
      cg_update_step<V, I, JAC><<<grid, block, 0, stream>>>(P, par);
    }
    launched += 2 * (uint64_t)upto;
    cudaError_t e = cudaMemcpyAsync(&active, &P.glob->active, sizeof(active), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(e);
  }
  cg_finish<V, I><<<grid, block, 0, stream>>>(P);
  launched += 1;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  (void)launched;
  if (!info) return SLA_OK;
  return read_info(P.ctl, P.glob, batch, stream, info);
}

}  // namespace

// Resident persistent kernel and cluster-resident kernel (sla_resident.cu).
template <typename V, typename I, bool JAC>
sla_status run_resident(Prob<V, I> P, cudaStream_t stream, sla_cg_info *info);
template <typename V, typename I, bool JAC>
sla_status run_cluster(Prob<V, I> P, int64_t batch, cudaStream_t stream, sla_cg_info *info);

namespace {

template <typename V, typename I, bool JAC>
sla_status run_cg(Prob<V, I> P, int unroll, int loop, cudaStream_t stream, sla_cg_info *info, int64_t batch) {
  const int dt = sizeof(V) == 8 ? SLA_F64 : SLA_F32;
  const int pc = JAC ? SLA_PRECOND_JACOBI : SLA_PRECOND_NONE;
  if (loop == SLA_LOOP_CLUSTER) {
    set_last_path(SLA_LOOP_CLUSTER);
    return run_cluster<V, I, JAC>(P, batch, stream, info);
  }
  if (loop == SLA_LOOP_AUTO && cluster_fits(P.n, batch, dt, pc)) {
    set_last_path(SLA_LOOP_CLUSTER);
    const sla_status st = run_cluster<V, I, JAC>(P, batch, stream, info);
    if (st != SLA_INVALID_ARG) return st;  // else the cluster could not be placed: next option
  }
  if (loop == SLA_LOOP_RESIDENT) {
    set_last_path(SLA_LOOP_RESIDENT);
    return run_resident<V, I, JAC>(P, stream, info);
  }
  if (loop == SLA_LOOP_AUTO && resident_fits(P.n, batch, dt, pc, P.maxit)) {
    set_last_path(SLA_LOOP_RESIDENT);
    const sla_status st = run_resident<V, I, JAC>(P, stream, info);
    if (st != SLA_INVALID_ARG) return st;  // else its blocks could not all be resident: next option
  }
  set_last_path(loop == SLA_LOOP_HOST ? SLA_LOOP_HOST : SLA_LOOP_GRAPH);
  const DeviceInfo di = device_info();
  Launch Lc;
  // TMA-staged SpMV step when every array it copies from is 16-byte aligned (per system too)
  const bool per_sys_ok = batch == 1 || (((size_t)P.n * sizeof(V)) % 16 == 0 &&
                                         ((size_t)P.val_stride * sizeof(V)) % 16 == 0);
  Lc.tma = tma_enabled() && per_sys_ok && aligned16(P.ci) && aligned16(P.val) && aligned16(P.x) &&
           aligned16(P.r) && aligned16(P.p[0]) && aligned16(P.p[1]) && (!JAC || aligned16(P.z));
  Lc.tma_smem = (unsigned)tma_smem_bytes<V>();
  static std::atomic<int> occ_u_cache{0}, occ_s_cache{0}, occ_t_cache{0};
  int occ_u = occ_u_cache.load(), occ_s = occ_s_cache.load(), occ_t = occ_t_cache.load();
  if (occ_u == 0) {
    occ_u = occupancy_blocks(Kernels<V, I, JAC>::update_step());
    occ_s = occupancy_blocks(Kernels<V, I, JAC>::spmv_step());
    void *ft = Kernels<V, I, JAC>::spmv_step_tma();
    occ_t = 0;
    if (cudaFuncSetAttribute(ft, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lc.tma_smem) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_t, ft, kTmaBlock, Lc.tma_smem) != cudaSuccess)
      occ_t = 0;
    cudaGetLastError();  // clear a refused attribute, if any
    occ_u_cache.store(occ_u);
    occ_s_cache.store(occ_s);
    occ_t_cache.store(occ_t);
  }
  if (occ_t < 1) Lc.tma = false;
  Lc.G_main = choose_G(P.n, batch, di.sms, occ_u);
  Lc.G_spmv = choose_G(P.n, batch, di.sms, Lc.tma ? occ_t : occ_s);
  P.G = Lc.G_main;
  if (unroll <= 0) unroll = kDefaultUnroll;
  if (unroll & 1) unroll += 1;  // the ping-pong parity of the body must repeat
  if (loop == SLA_LOOP_HOST) return run_cg_host_loop<V, I, JAC>(P, Lc, unroll, stream, info, batch);

  // the graph's shape; the problem itself goes in as node arguments
  const int shape[8] = {(int)sizeof(V), (int)sizeof(I), (int)JAC, (int)Lc.tma, Lc.G_main, Lc.G_spmv,
                        (int)std::min<int64_t>(P.batch, INT32_MAX), unroll};
  std::vector<char> key((const char *)shape, (const char *)shape + sizeof(shape));
  int dev = di.dev;
  key.insert(key.end(), (char *)&dev, (char *)&dev + sizeof(dev));
  std::vector<char> pargs((const char *)&P, (const char *)&P + sizeof(P));

  {
    std::lock_guard<std::mutex> lk(g_mu);
    GraphEntry *hit = nullptr;
    for (auto &en : g_cache)
      if (en.key == key) {
        hit = &en;
        break;
      }
    if (hit && hit->args != pargs) {
      if (update_graph<V, I, JAC>(P, Lc, unroll, *hit) == cudaSuccess) {
        hit->args = pargs;
        ++g_updates;
      } else {  // arguments not replaceable here: rebuild this entry
        cudaGetLastError();
        cudaGraphExecDestroy(hit->exec);
        cudaGraphDestroy(hit->graph);
        g_cache.erase(g_cache.begin() + (hit - g_cache.data()));
        hit = nullptr;
      }
    }
    if (!hit) {
      GraphEntry en;
      en.key = key;
      en.args = pargs;
      cudaError_t e = build_graph<V, I, JAC>(P, Lc, unroll, en);
      if (e != cudaSuccess) return fail(e);
      ++g_builds;
      if (g_cache.size() >= kCacheCap) {
        auto it = std::min_element(g_cache.begin(), g_cache.end(),
                                   [](const GraphEntry &a, const GraphEntry &b) { return a.stamp < b.stamp; });
        cudaGraphExecDestroy(it->exec);
        cudaGraphDestroy(it->graph);
        g_cache.erase(it);
      }
      g_cache.push_back(std::move(en));
      hit = &g_cache.back();
    }
    hit->stamp = ++g_stamp;
    cudaError_t e = cudaGraphLaunch(hit->exec, stream);
    if (e != cudaSuccess) return fail(e);
  }
  if (!info) return SLA_OK;
  return read_info(P.ctl, P.glob, batch, stream, info);
}

template <typename V, typename I>
sla_status dispatch_precond(const Prob<V, I> &P, const sla_cg_opts *o, cudaStream_t st, sla_cg_info *info,
                            int64_t batch) {
  if (o->precond == SLA_PRECOND_JACOBI) return run_cg<V, I, true>(P, o->unroll, o->loop, st, info, batch);
  return run_cg<V, I, false>(P, o->unroll, o->loop, st, info, batch);
}

template <typename V, typename I>
Prob<V, I> make_prob(const sla_csr *A, int64_t batch, const void *values, int64_t val_stride, const void *b,
                     const void *x0, const sla_cg_opts *o, void *x, double *history, void *ws, bool jacobi,
                     bool halo_ws) {
  Prob<V, I> P;
  memset(&P, 0, sizeof(P));
  Layout L = make_layout(A->n, batch, sizeof(V), jacobi, halo_ws);
  char *w = (char *)ws;
  P.rp = (const I *)A->row_ptr;
  P.ci = A->col_idx;
  P.val = (const V *)values;
  P.b = (const V *)b;
  P.x0 = (const V *)x0;
  P.x = (V *)x;
  P.r = (V *)(w + L.r);
  P.p[0] = (V *)(w + L.p0);
  P.p[1] = (V *)(w + L.p1);
  P.q = (V *)(w + L.q);
  P.dinv = jacobi ? (V *)(w + L.dinv) : nullptr;
  P.z = jacobi ? (V *)(w + L.z) : nullptr;
  P.partials = (double *)(w + L.partials);
  P.ctl = (Ctl *)(w + L.ctl);
  P.glob = (Glob *)(w + L.glob);
  P.halo = halo_ws ? (uint32_t *)(w + L.halo) : nullptr;
  P.history = history;
  P.val_stride = val_stride;
  P.nnz = A->nnz;
  P.maxit = o->maxit;
  P.rtol = o->rtol;
  P.n = (int32_t)A->n;
  P.batch = (int32_t)batch;
  return P;
}

}  // namespace

sla_status cg_entry(const sla_csr *A, int64_t batch, const void *values, int64_t val_stride, const void *b,
                    const void *x0, const sla_cg_opts *o, void *x, sla_cg_info *info, double *history, void *ws,
                    cudaStream_t st, bool halo_ws) {
  const bool jac = o->precond == SLA_PRECOND_JACOBI;
  if (A->dtype == SLA_F64) {
    if (A->rowptr_type == SLA_I64)
      return dispatch_precond(make_prob<double, int64_t>(A, batch, values, val_stride, b, x0, o, x, history, ws, jac, halo_ws),
                              o, st, info, batch);
    return dispatch_precond(make_prob<double, int32_t>(A, batch, values, val_stride, b, x0, o, x, history, ws, jac, halo_ws),
                            o, st, info, batch);
  }
  if (A->rowptr_type == SLA_I64)
    return dispatch_precond(make_prob<float, int64_t>(A, batch, values, val_stride, b, x0, o, x, history, ws, jac, halo_ws),
                            o, st, info, batch);
  return dispatch_precond(make_prob<float, int32_t>(A, batch, values, val_stride, b, x0, o, x, history, ws, jac, halo_ws),
                          o, st, info, batch);
}

size_t workspace_bytes(int64_t n, int64_t batch, int dtype, int precond) {
  return make_layout(n, batch, dtype == SLA_F64 ? 8 : 4, precond == SLA_PRECOND_JACOBI).total;
}

}  // namespace sla

extern "C" sla_status sla_graph_cache_stats(int64_t *entries, int64_t *builds, int64_t *updates) {
  std::lock_guard<std::mutex> lk(sla::g_mu);
  if (entries) *entries = (int64_t)sla::g_cache.size();
  if (builds) *builds = (int64_t)sla::g_builds;
  if (updates) *updates = (int64_t)sla::g_updates;
  return SLA_OK;
}

extern "C" sla_status sla_set_spmv_variant(int32_t variant) {
  if (variant != SLA_SPMV_PLAIN && variant != SLA_SPMV_TMA) return SLA_INVALID_ARG;
  sla::g_spmv_variant.store(variant);
  return SLA_OK;
}
