"""Benchmark of the differentiable CSR CG solve (forward + adjoint backward) on GB300.

One step = one pass of the whole hot path over one synthetic system: the CG solve
A x = b (sla_cg_solve) and the adjoint backward (sla_cg_adjoint: A lambda = g,
grad_b = lambda, grad_values = -lambda_i x_j on the pattern).  The default workload
is the 1M-DOF 2D Poisson system in fp64 (m = 1000, nnz = 4,996,000), CG rtol 1e-8,
b ~ N(0,1) seed 0, g ~ N(0,1) seed 1.

Metric: CG iterations per second over the whole job (forward + adjoint iterations of
all ranks / the max-over-ranks device time of the timed steps), plus the effective HBM
GB/s of the fused CG iteration against the measured copy bandwidth, and the adjoint ms.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}] [--config NAME]

NAME: poisson64, poisson1000 (default), diffusion128_batch64, diffusion4096_jacobi,
poisson13000_int64 (short aliases config1 .. config5); eig_poisson: the smallest eigenpair
of the 1M-DOF Poisson matrix by inverse iteration on the CG plus its eigenvalue gradient;
convdiff1000_bicgstab: the 1M-DOF convection-diffusion operator (non-symmetric) by BiCGStab,
forward and adjoint.

With N > 1 the script runs under torch.distributed.run; every rank solves its own
independent system of the same size (replicas, weak scaling).  --dist splits one system
across the ranks instead (row blocks with halo exchange, strong scaling).  --impl reference times the fp64 CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CG iters/sec and HBM GB/s (% of roofline), 1M-DOF 2D Poisson fp64; adjoint ms"


def b_iter(n, nnz, s_v, s_p, jacobi):
    """Algorithmic bytes of one fused CG iteration: matrix stream + row pointers + V vector passes."""
    V = 11 if jacobi else 9
    return nnz * (s_v + 4) + (n + 1) * s_p + V * n * s_v


def b_iter_batched(batch, n, nnz, s_v):
    """Algorithmic bytes of one batched iteration: every system's values and vectors, the shared
    pattern (col_idx, int32 row_ptr) read once."""
    return batch * (nnz * s_v + 9 * n * s_v) + nnz * 4 + (n + 1) * 4


def b_iter_bicgstab(n, nnz, s_v, s_p):
    """Algorithmic bytes of one BiCGStab iteration: two matrix streams (A p and A s) and 17 vector
    passes (p and A p: r, p_prev, v_prev, rhat read, p, v written; s and A s: r, v read, s, t
    written; update: x, p, s, t, rhat read, x, r written)."""
    return 2 * (nnz * (s_v + 4) + (n + 1) * s_p) + 17 * n * s_v


def flops_iter_bicgstab(n, nnz):
    """fp64 flops of one BiCGStab iteration, 2 per multiply-add: the products A p and A s (2 nnz
    each) and 12 multiply-adds per row (p 2, s 1, x 2, r 1, and the dot products rhat.v, s.s, t.s,
    t.t, rhat.r, r.r)."""
    return 4 * nnz + 24 * n


def b_gradvalues(n, nnz, s_v, s_p):
    """One grad_values pass: col_idx read + gv write, row pointers, lambda and x reads."""
    return nnz * (s_v + 4) + (n + 1) * s_p + 2 * n * s_v


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def fp64_peak_tflops(clocks=None):
    """fp64 FMA peak of GB300: 152 SMs x 2 FMA per clock (1.25 TFLOP/s nominal) at the max SM clock."""
    mhz = 2070.0
    if clocks and clocks.get("sm_max_mhz"):
        mhz = float(clocks["sm_max_mhz"])
    return 152 * 2 * 2 * mhz * 1e6 / 1e12


# The sources each engine's CG kernels are compiled from: a traffic record in profiles/traffic.json
# stays valid while these files are unchanged.  Host-side files (argument checks, entry points),
# the gradient and eigenvalue kernels and the other engines' files hold none of them.
KERNEL_SOURCES = {
    "cluster": ("sla_common.cuh", "sla_onchip.cuh", "sla_cluster.cu"),
    "resident": ("sla_common.cuh", "sla_grid.cuh", "sla_onchip.cuh", "sla_resident.cu"),
    "streaming": ("sla_common.cuh", "sla_tma.cuh", "sla_stream.cuh"),
    "bicgstab": ("sla_common.cuh", "sla_grid.cuh", "sla_bicgstab.cu"),
}
ENGINE_OF = {"config1": "cluster", "config3": "cluster", "config2": "resident", "config4": "streaming",
             "config5": "streaming", "convdiff1000_bicgstab": "bicgstab"}


def csrc_sha256(engine):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[engine]:
        h.update(name.encode())
        with open(os.path.join(ROOT, "differentiable_sparse_iterative_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def canonical_name(name):
    from workloads import canonical_name as cn
    return cn(name)


def profiled_traffic(config):
    """DRAM bytes per CG iteration from the committed ncu summary, or None when the kernel
    sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(config)
    except (OSError, ValueError):
        return None
    if not rec or config not in ENGINE_OF or rec.get("csrc_sha256") != csrc_sha256(ENGINE_OF[config]):
        return None
    return rec


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def aggregate_over_ranks(seconds, iters, world, device=None):
    """Whole-job numbers of a replicated run: the slowest rank's time and all ranks' iterations.

    Each rank solves its own system (no exchange on the data path); the job's throughput is the
    sum of iterations over the max time.  With world == 1 this is the identity."""
    if world <= 1:
        return float(seconds), float(iters)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    it = torch.tensor([float(iters)], dtype=torch.float64, device=device)
    dist.all_reduce(it, op=dist.ReduceOp.SUM)
    return float(t.item()), float(it.item())


def flush_l2(buf):
    buf.zero_()  # a write larger than the 129 MB L2 evicts the previous step's lines


def run_ours(args, rank, world, local_rank):
    import torch
    import differentiable_sparse_iterative_gb300 as sla
    from workloads import config_by_name

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = config_by_name(args.config, **({"m": args.grid_m} if args.grid_m else {}))
    precond = w.precond
    jac = precond == 1
    batched = w.batch > 0
    if batched:
        return run_batched(args, w, dev, rank, world)
    # the bench's own L2-flush buffer first: the device memory counted below is the step's alone
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    mem_base = torch.cuda.memory_allocated(dev)
    A = sla.CSRMatrix.from_numpy(w.A.row_ptr, w.A.col_idx, w.A.values, dev)
    b = torch.from_numpy(w.b).to(dev)
    g_np = w.g if w.g is not None else np.random.default_rng(1).standard_normal(w.A.n)
    g = torch.from_numpy(g_np).to(dev)
    n, nnz = w.A.n, w.A.nnz
    s_v, s_p = 8, w.A.row_ptr.dtype.itemsize
    ws = torch.empty(sla.sla_cg_workspace_bytes(n, 1, torch.float64, precond), dtype=torch.uint8, device=dev)
    x = torch.empty(n, dtype=torch.float64, device=dev)
    gb = torch.empty(n, dtype=torch.float64, device=dev)
    gv = torch.empty(nnz, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    loop = {"auto": sla.SLA_LOOP_AUTO, "cluster": sla.SLA_LOOP_CLUSTER, "resident": sla.SLA_LOOP_RESIDENT,
            "graph": sla.SLA_LOOP_GRAPH,
            "host": sla.SLA_LOOP_HOST}[args.loop]

    def step():
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        _, fi, _ = sla.sla_cg_solve(A, b, rtol=w.rtol, maxit=w.maxit, precond=precond, x=x, workspace=ws,
                                    loop=loop)
        e1.record(stream)
        _, _, ai = sla.sla_cg_adjoint(A, x, g, rtol=w.rtol, maxit=w.maxit, precond=precond, grad_b=gb,
                                      grad_values=gv, workspace=ws, loop=loop)
        e2.record(stream)
        return e0, e1, e2, fi, ai

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = sla.sla_launch_count()
    recs = []
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush_l2(flush)
            recs.append(step())
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    launches = sla.sla_launch_count() - launches0
    fwd_ms = [r[0].elapsed_time(r[1]) for r in recs]
    adj_ms = [r[1].elapsed_time(r[2]) for r in recs]
    iters_f = [r[3].iters for r in recs]
    iters_a = [r[4].iters for r in recs]
    status = {r[3].status for r in recs} | {r[4].status for r in recs}
    step_ms = [f + a for f, a in zip(fwd_ms, adj_ms)]
    tot_s = sum(step_ms) / 1e3
    tot_iters = sum(iters_f) + sum(iters_a)
    # device memory of forward + adjoint: matrix, b, g, x, grad_b, grad_values and the O(n) workspace
    peak_mem = torch.cuda.max_memory_allocated(dev) - mem_base
    ws_mb = ws.numel() / 2**20

    tot_s_all, tot_iters_all = aggregate_over_ranks(tot_s, tot_iters, world, dev)

    Bi = b_iter(n, nnz, s_v, s_p, jac)
    Bg = b_gradvalues(n, nnz, s_v, s_p)
    peak, peak_kind = measured_peaks()
    # fused CG iteration (spmv_step + update_step): bytes per iteration / forward time per iteration
    fwd_s = sum(fwd_ms) / 1e3
    achieved = Bi * sum(iters_f) / fwd_s / 1e9
    tr = None if args.grid_m else profiled_traffic(canonical_name(args.config))  # counters are for the full-size workload
    clocks = clk.summary()
    path = recs[-1][3].path
    kernel_name = {"resident": "cg_resident (one persistent cooperative kernel per solve)",
                   "cluster": "cg_cluster (one thread-block cluster per system)",
                   "graph": "cg_spmv_step + cg_update_step (CUDA graph loop)",
                   "host": "cg_spmv_step + cg_update_step (host loop)"}.get(path, path)
    # fp64 issue roofline: algorithmic fp64 flops of one iteration against 152 SMs x 2 FMA/clk
    flops_it = 2 * nnz + (13 if jac else 10) * n
    fp64_peak = fp64_peak_tflops(clocks)
    fp64_ach = flops_it * sum(iters_f) / fwd_s / 1e12

    grad_k = grad_kernel_timing(A, gb, x, gv, flush, stream, sla, torch, peak, Bg)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, dev, precond, sla, torch)

    out = {
        "metric": METRIC, "value": tot_iters_all / tot_s_all, "unit": "iters/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators; no dataset on the pages)",
        "config": {"workload": w.name, "n": n, "nnz": nnz, "rtol": w.rtol, "precond": "jacobi" if jac else "none",
                   "step": "forward CG solve + adjoint (grad_b, grad_values)",
                   "l2": "flushed between steps (256 MB write); within a solve the iterations reuse L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "loop": args.loop},
        "iters_forward": statistics.mean(iters_f), "iters_adjoint": statistics.mean(iters_a),
        "time_to_tolerance_ms": statistics.mean(fwd_ms), "adjoint_ms": statistics.mean(adj_ms),
        "status": sorted(status),
        "effective_gbs_step": (Bi * tot_iters + Bg * args.steps) / tot_s / 1e9,
        "peak_mem_mb": peak_mem / 2**20,
        "workspace_mb": ws_mb,
        "path": path,
        "fp64": {"achieved_tflops": fp64_ach, "peak_tflops": fp64_peak, "frac": fp64_ach / fp64_peak,
                 "flops_per_iter": flops_it,
                 "peak_basis": "152 SMs x 2 fp64 FMA/clock x 2 flops x max SM clock"},
        "roofline": {"kernel": kernel_name, "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind,
                     "bytes_per_iter": Bi,
                     "traffic": (tr["dram_bytes_per_iter"] if tr else None),
                     "traffic_unit": "DRAM bytes per CG iteration (ncu dram__bytes_read + write)",
                     "traffic_source": (tr.get("source") if tr else None)},
        "grad_values_roofline": grad_k,
        "gpu_launches": int(launches),
        "wall_s": wall,
        "clocks": clocks,
    }
    if e2e:
        out["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_iters)
    return out


def grad_kernel_timing(A, lam, x, gv, flush, stream, sla, torch, peak, Bg, reps=20):
    """grad_values_kernel alone, each launch after an L2 flush (a 256 MB write): per-launch CUDA
    events (the flush keeps the GPU busy while the launch is enqueued), and the difference between
    reps x (flush + kernel) and reps x flush.  Beside it, for scale, PyTorch's index_select over the
    same col_idx (x gathered per entry, one value written per entry: the kernel's access pattern
    without the row factor) timed the same way: what a plain library gather reaches at this size."""
    ci = A.col_idx
    try:
        torch.index_select(x, 0, ci[:1])
    except (RuntimeError, TypeError):  # a PyTorch without 32-bit indices: 64-bit ones, counted as such
        ci = ci.long()
    sel = torch.empty(A.nnz, dtype=x.dtype, device=x.device)

    def timed(fn):
        per = []
        for _ in range(reps):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            per.append((a, b))
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        for _ in range(reps):
            flush_l2(flush)
            fn()
        e[1].record(stream)
        for _ in range(reps):
            flush_l2(flush)
        e[2].record(stream)
        torch.cuda.synchronize()
        ev_ms = statistics.mean(a.elapsed_time(b) for a, b in per)
        diff_ms = (e[0].elapsed_time(e[1]) - e[1].elapsed_time(e[2])) / reps
        return ev_ms, diff_ms

    import ctypes
    cs = sla._csr_struct(A)  # arguments marshalled once: each launch is one C call
    lib, sh = sla.lib(), stream.cuda_stream
    lp, xp, gp = lam.data_ptr(), x.data_ptr(), gv.data_ptr()

    def kernel():
        assert lib.sla_grad_values(ctypes.byref(cs), lp, xp, gp, sh) == 0

    for _ in range(3):  # warm-up
        kernel()
        torch.index_select(x, 0, ci, out=sel)
    k_ev, k_diff = timed(kernel)
    g_ev, g_diff = timed(lambda: torch.index_select(x, 0, ci, out=sel))
    Bsel = A.nnz * (ci.element_size() + x.element_size()) + A.n * x.element_size()  # col_idx, values written, x
    return {"kernel": "grad_values_kernel", "bound": "hbm", "unit": "GB/s", "peak": peak,
            "bytes_per_launch": Bg,
            "achieved": Bg / (k_ev / 1e3) / 1e9, "frac": Bg / (k_ev / 1e3) / 1e9 / peak, "us_events": k_ev * 1e3,
            "achieved_flush_subtracted": Bg / (k_diff / 1e3) / 1e9,
            "frac_flush_subtracted": Bg / (k_diff / 1e3) / 1e9 / peak, "us_flush_subtracted": k_diff * 1e3,
            "gather_floor": {"op": "torch.index_select(x, 0, col_idx)", "bytes_per_launch": Bsel,
                             "us_events": g_ev * 1e3, "frac": Bsel / (g_ev / 1e3) / 1e9 / peak,
                             "us_flush_subtracted": g_diff * 1e3,
                             "frac_flush_subtracted": Bsel / (g_diff / 1e3) / 1e9 / peak},
            "timing": f"{reps} launches, each after a 256 MB L2 flush, CUDA events"}


def run_dist(args, rank, world, local_rank):
    """One system split across the ranks (row blocks of whole grid rows, halo exchange, sums over ranks:
    the distributed layer): forward solve + adjoint per step, timed on every rank, max over ranks.
    Strong scaling: the system is the same for every N."""
    import torch
    import torch.distributed as dist
    from differentiable_sparse_iterative_gb300 import distributed as D
    from workloads import config_by_name

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = config_by_name(args.config, **({"m": args.grid_m} if args.grid_m else {}))
    if w.batch > 0:
        raise SystemExit("--dist takes a single-system workload")
    m = int(w.meta.get("m", 1))
    bounds = D.partition_rows(w.A.row_ptr, world, m)
    blk = D.local_block(w.A.row_ptr, w.A.col_idx, w.A.values, bounds, rank)
    solver = D.DistCG(blk, D.TorchComm(), device=dev)
    g_np = w.g if w.g is not None else np.random.default_rng(1).standard_normal(w.A.n)
    b = torch.from_numpy(w.b[blk.lo:blk.hi].copy()).to(dev)
    g = torch.from_numpy(g_np[blk.lo:blk.hi].copy()).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        x, fi, _ = solver.solve(b, rtol=w.rtol, maxit=w.maxit, precond=w.precond)
        e1.record(stream)
        _, _, ai = solver.adjoint(x, g, rtol=w.rtol, maxit=w.maxit, precond=w.precond)
        e2.record(stream)
        return e0, e1, e2, fi, ai

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    recs = []
    with ClockSampler(local_rank) as clk:
        for _ in range(args.steps):
            flush_l2(flush)
            recs.append(step())
        torch.cuda.synchronize()
    dist.barrier()
    fwd_ms = [r[0].elapsed_time(r[1]) for r in recs]
    adj_ms = [r[1].elapsed_time(r[2]) for r in recs]
    its = sum(r[3].iters + r[4].iters for r in recs)
    t = torch.tensor([sum(fwd_ms) + sum(adj_ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tot_s = float(t.item()) / 1e3
    n, nnz = w.A.n, w.A.nnz
    Bi = b_iter(n, nnz, 8, w.A.row_ptr.dtype.itemsize, w.precond == 1)
    peak, peak_kind = measured_peaks()
    achieved = Bi * sum(r[3].iters for r in recs) / (sum(fwd_ms) / 1e3) / 1e9
    return {
        "metric": METRIC, "value": its / tot_s, "unit": "iters/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators; no dataset on the pages)",
        "config": {"workload": w.name, "n": n, "nnz": nnz, "rtol": w.rtol,
                   "precond": "jacobi" if w.precond == 1 else "none",
                   "step": "forward CG solve + adjoint (grad_b, grad_values), one system over all ranks",
                   "l2": "flushed between steps (256 MB write)",
                   "parallelism": f"row blocks x{world} (halo exchange, all-gathered partial sums)"},
        "iters_forward": statistics.mean(r[3].iters for r in recs),
        "iters_adjoint": statistics.mean(r[4].iters for r in recs),
        "time_to_tolerance_ms": statistics.mean(fwd_ms), "adjoint_ms": statistics.mean(adj_ms),
        "status": sorted({r[3].status for r in recs} | {r[4].status for r in recs}),
        "path": "distributed",
        "roofline": {"kernel": "sla_dist_* steps (job-wide algorithmic bytes over the job's peak)", "bound": "hbm",
                     "achieved": achieved, "peak": peak * world, "unit": "GB/s",
                     "frac": achieved / (peak * world), "peak_kind": peak_kind, "bytes_per_iter": Bi,
                     "traffic": None},
        "rows_per_rank": [int(bounds[q + 1] - bounds[q]) for q in range(world)],
        "clocks": clk.summary(),
    }


def run_batched(args, w, dev, rank, world):
    """Batched shared-pattern workload (config 3): forward + adjoint of all systems per step.
    The metric counts system-iterations (each system's CG iterations, summed over the batch)."""
    import torch
    import differentiable_sparse_iterative_gb300 as sla
    dt = torch.float32 if w.dtype == "f32" else torch.float64
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    mem_base = torch.cuda.memory_allocated(dev)
    P = sla.CSRMatrix.from_numpy(w.A.row_ptr, w.A.col_idx, w.A.values.astype(np.float32 if dt == torch.float32
                                                                              else np.float64), dev)
    vals = torch.from_numpy(w.values_b).to(dev)
    b = torch.from_numpy(w.b).to(dev)
    g = torch.from_numpy(w.g).to(dev)
    B, n, nnz = w.batch, w.A.n, w.A.nnz
    loop = {"auto": sla.SLA_LOOP_AUTO, "cluster": sla.SLA_LOOP_CLUSTER, "resident": sla.SLA_LOOP_RESIDENT,
            "graph": sla.SLA_LOOP_GRAPH,
            "host": sla.SLA_LOOP_HOST}[args.loop]
    stream = torch.cuda.current_stream(dev)

    def step():
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        x, fi, _ = sla.sla_cg_solve_batched(P, vals, b, rtol=w.rtol, maxit=w.maxit, precond=w.precond, loop=loop)
        e1.record(stream)
        _, _, ai = sla.sla_cg_adjoint_batched(P, vals, x, g, rtol=w.rtol, maxit=w.maxit, precond=w.precond,
                                              loop=loop)
        e2.record(stream)
        return e0, e1, e2, fi, ai

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    launches0 = sla.sla_launch_count()
    recs = []
    with ClockSampler(local_rank_of(dev)) as clk:
        for _ in range(args.steps):
            flush_l2(flush)
            recs.append(step())
        torch.cuda.synchronize()
    launches = sla.sla_launch_count() - launches0
    peak_mem = torch.cuda.max_memory_allocated(dev) - mem_base
    fwd_ms = [r[0].elapsed_time(r[1]) for r in recs]
    adj_ms = [r[1].elapsed_time(r[2]) for r in recs]
    it_f = [sum(i.iters for i in r[3]) for r in recs]
    it_a = [sum(i.iters for i in r[4]) for r in recs]
    tot_s = (sum(fwd_ms) + sum(adj_ms)) / 1e3
    s_v = 4 if dt == torch.float32 else 8
    peak, peak_kind = measured_peaks()
    max_it = [max(i.iters for i in r[3]) for r in recs]
    tr = None if args.grid_m else profiled_traffic(canonical_name(args.config))  # counters are for the full-size workload
    Bi_batch = b_iter_batched(B, n, nnz, s_v)
    achieved = Bi_batch * sum(max_it) / (sum(fwd_ms) / 1e3) / 1e9
    return {
        "metric": METRIC, "value": (sum(it_f) + sum(it_a)) / tot_s, "unit": "system-iters/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": (sum(fwd_ms) + sum(adj_ms)) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32" if s_v == 4 else "f64",
        "data": "synthetic (seeded generators; no dataset on the pages)",
        "config": {"workload": w.name, "n": n, "nnz": nnz, "batch": B, "rtol": w.rtol, "loop": args.loop,
                   "step": "batched forward CG + batched adjoint"},
        "iters_forward_max": statistics.mean(max_it), "time_to_tolerance_ms": statistics.mean(fwd_ms),
        "adjoint_ms": statistics.mean(adj_ms),
        "peak_mem_mb": peak_mem / 2**20,
        "path": recs[-1][3][0].path,
        "roofline": {"kernel": {"cluster": "cg_cluster (one thread-block cluster per system)",
                                "graph": "cg_spmv_step + cg_update_step, one grid row per system (CUDA graph loop)",
                                "host": "cg_spmv_step + cg_update_step, one grid row per system (host loop)"}.get(
                                    recs[-1][3][0].path, "batched CG iteration"), "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind, "bytes_per_iter": Bi_batch,
                     "traffic": (tr["dram_bytes_per_iter"] if tr else None),
                     "traffic_unit": "DRAM bytes per batched CG iteration (ncu dram__bytes_read + write)",
                     "traffic_source": (tr.get("source") if tr else None)},
        "gpu_launches": int(launches), "clocks": clk.summary(),
        **({} if args.no_e2e else {"e2e": run_e2e_batched(args, w, dev, sla, torch, it_f[-1] + it_a[-1])}),
    }


def run_e2e_batched(args, w, dev, sla, torch, sys_iters_per_step):
    """The batched step through the public autograd API (solve_batched + backward): pattern, values
    [S, nnz], b and g from pinned host memory, x and both gradients read back, every step."""
    h = {k: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
         for k, a in (("rp", w.A.row_ptr), ("ci", w.A.col_idx), ("v", w.values_b), ("b", w.b), ("g", w.g))}
    o_x = torch.empty(w.b.shape, dtype=h["b"].dtype).pin_memory()
    o_gb = torch.empty(w.b.shape, dtype=h["b"].dtype).pin_memory()
    o_gv = torch.empty(w.values_b.shape, dtype=h["v"].dtype).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in (o_x, o_gb, o_gv))
    stream = torch.cuda.current_stream(dev)

    def step():
        rp, ci = h["rp"].to(dev, non_blocking=True), h["ci"].to(dev, non_blocking=True)
        v = h["v"].to(dev, non_blocking=True).requires_grad_(True)
        b = h["b"].to(dev, non_blocking=True).requires_grad_(True)
        g = h["g"].to(dev, non_blocking=True)
        x = sla.solve_batched(rp, ci, v, b, rtol=w.rtol, maxit=w.maxit, precond=w.precond)
        x.backward(g)
        o_x.copy_(x.detach(), non_blocking=True)
        o_gb.copy_(b.grad, non_blocking=True)
        o_gv.copy_(v.grad, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    return {"value": sys_iters_per_step * args.steps / total, "unit": "system-iters/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "api": "differentiable_sparse_iterative_gb300.solve_batched + backward"}


def local_rank_of(dev):
    return dev.index if dev.index is not None else 0


def run_e2e(args, w, dev, precond, sla, torch, method="cg"):
    """The same step through the public autograd API, inputs from pinned host memory, results back."""
    h_rp = torch.from_numpy(w.A.row_ptr).pin_memory()
    h_ci = torch.from_numpy(w.A.col_idx).pin_memory()
    h_v = torch.from_numpy(w.A.values).pin_memory()
    h_b = torch.from_numpy(w.b).pin_memory()
    g_np = w.g if w.g is not None else np.random.default_rng(1).standard_normal(w.A.n)
    h_g = torch.from_numpy(g_np).pin_memory()
    o_x = torch.empty(w.A.n, dtype=torch.float64).pin_memory()
    o_gb = torch.empty(w.A.n, dtype=torch.float64).pin_memory()
    o_gv = torch.empty(w.A.nnz, dtype=torch.float64).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (h_rp, h_ci, h_v, h_b, h_g))
    d2h = sum(t.numel() * t.element_size() for t in (o_x, o_gb, o_gv))
    stream = torch.cuda.current_stream(dev)
    iters = []

    def step():
        rp = h_rp.to(dev, non_blocking=True)
        ci = h_ci.to(dev, non_blocking=True)
        v = h_v.to(dev, non_blocking=True).requires_grad_(True)
        b = h_b.to(dev, non_blocking=True).requires_grad_(True)
        g = h_g.to(dev, non_blocking=True)
        A = sla.CSRMatrix(rp, ci, v)
        xx = sla.solve(A, b, rtol=w.rtol, maxit=w.maxit, precond=precond, method=method)
        xx.backward(g)
        o_x.copy_(xx.detach(), non_blocking=True)
        o_gb.copy_(b.grad, non_blocking=True)
        o_gv.copy_(v.grad, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    mem_base = torch.cuda.memory_allocated(dev)
    total = 0.0
    for _ in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1) / 1e3
    peak_mem = torch.cuda.max_memory_allocated(dev) - mem_base
    # iterations of the autograd path equal those of the direct calls on the same data
    Ad = sla.CSRMatrix(h_rp.to(dev), h_ci.to(dev), h_v.to(dev))
    if method == "bicgstab":
        _, fi, _ = sla.sla_bicgstab_solve(Ad, h_b.to(dev), rtol=w.rtol, maxit=w.maxit)
        _, _, ai = sla.sla_bicgstab_adjoint(Ad, o_x.to(dev), h_g.to(dev), rtol=w.rtol, maxit=w.maxit)
    else:
        _, fi, _ = sla.sla_cg_solve(Ad, h_b.to(dev), rtol=w.rtol, maxit=w.maxit, precond=precond)
        _, _, ai = sla.sla_cg_adjoint(Ad, o_x.to(dev), h_g.to(dev), rtol=w.rtol, maxit=w.maxit, precond=precond)
    per_step_iters = fi.iters + ai.iters
    return {"value": per_step_iters * args.steps / total, "unit": "iters/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "api": f"differentiable_sparse_iterative_gb300.solve(method={method!r}) + backward",
            "peak_mem_mb": peak_mem / 2**20}


def cpu_baseline(w, iters):
    """The fp64 oracle as it stands, multi-core build on every host core, on a bounded sample:
    `iters` forward CG iterations plus `iters` adjoint iterations on the same system (iters = 0:
    sized from a short probe to about 15 s of host time)."""
    import oracle
    lib = oracle.load_parallel()
    cores = lib.orc_threads(0)
    g = w.g if w.g is not None else np.random.default_rng(1).standard_normal(w.A.n)
    fwd, adj, what = _oracle_pair(w, lib)
    if iters <= 0:
        t0 = time.perf_counter()
        fwd(20)
        per_it = (time.perf_counter() - t0) / 20
        iters = int(min(20000, max(100, 7.5 / max(per_it, 1e-6))))
    t0 = time.perf_counter()
    f = fwd(iters)
    a = adj(f["x"], g, iters)
    dt = time.perf_counter() - t0
    return {"value": (f["iters"] + a["iters"]) / dt, "unit": "iters/s", "cores": cores, "kind": "oracle",
            "sample": f"{w.name}: {f['iters']} forward + {a['iters']} adjoint {what} iterations (rtol 0, at most "
                      f"{iters} each) and one grad_values pass, {dt:.1f} s on {cores} host cores (the oracle's "
                      f"multi-core build)"}


def _oracle_pair(w, lib):
    """The oracle's forward solve and adjoint for a workload, as functions of the iteration count."""
    import oracle
    A = w.A
    if w.meta.get("method") == "bicgstab":
        return (lambda k: oracle.bicgstab(A.row_ptr, A.col_idx, A.values, w.b, rtol=0.0, maxit=k, lib=lib),
                lambda x, g, k: oracle.bicgstab_adjoint(A.row_ptr, A.col_idx, A.values, x, g, rtol=0.0, maxit=k,
                                                        lib=lib),
                "BiCGStab")
    return (lambda k: oracle.cg(A.row_ptr, A.col_idx, A.values, w.b, rtol=0.0, maxit=k, precond=w.precond, lib=lib),
            lambda x, g, k: oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, x, g, rtol=0.0, maxit=k,
                                              precond=w.precond, lib=lib),
            "CG")


EIG_METRIC = "smallest eigenpair (inverse iteration on CG) + eigenvalue gradient, 2D Poisson fp64: CG iters/sec"


def b_eig_grad(n, nnz, s_v, s_p):
    """One eigenvalue-gradient pass (one eigenvector): col_idx read + gv write, row pointers, v read once
    (the gathers of v[col] assumed served by cache)."""
    return nnz * (s_v + 4) + (n + 1) * s_p + n * s_v


def run_eig(args, rank, world, local_rank):
    """Eigenvalue workload: the smallest eigenpair of the 2D Poisson matrix by inverse iteration
    (each step one inner CG solve) and the Hellmann-Feynman gradient v_i v_j on the pattern.  The
    metric counts the inner CG iterations; the eigen-solve's time includes the host-driven outer
    loop (one scalar read per step)."""
    import torch
    import differentiable_sparse_iterative_gb300 as sla
    from workloads import poisson_5pt, config_by_name
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    m = args.grid_m or 1000
    A_np = poisson_5pt(m)
    n, nnz = A_np.n, A_np.nnz
    s_v, s_p = 8, A_np.row_ptr.dtype.itemsize
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    A = sla.CSRMatrix.from_numpy(A_np.row_ptr, A_np.col_idx, A_np.values, dev)
    ws = torch.empty(sla.sla_eig_workspace_bytes(n, torch.float64), dtype=torch.uint8, device=dev)
    gv = torch.empty(nnz, dtype=torch.float64, device=dev)
    ones = torch.ones(n, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    tol = 1e-10

    def step():
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        mu, v, info = sla.sla_eig_smallest(A, v0=ones, tol=tol, workspace=ws)
        e1.record(stream)
        sla.sla_eig_grad_values(A, v, out=gv)
        e2.record(stream)
        return e0, e1, e2, info

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = sla.sla_launch_count()
    recs = []
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush_l2(flush)
            recs.append(step())
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    launches = sla.sla_launch_count() - launches0
    eig_ms = [r[0].elapsed_time(r[1]) for r in recs]
    grad_ms = [r[1].elapsed_time(r[2]) for r in recs]
    # The gradient kernel alone: in a step it starts after the eigen-solve's final synchronisation,
    # so its interval there includes the host's launch latency.  Here each launch follows an L2
    # flush that keeps the GPU busy while the host enqueues it (arguments marshalled once).
    import ctypes
    cs = sla._csr_struct(A)
    v_last = sla.sla_eig_smallest(A, v0=ones, tol=tol, workspace=ws)[1]
    lib, sh = sla.lib(), stream.cuda_stream
    kern_ms = []
    for _ in range(20):
        flush_l2(flush)
        ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ka.record(stream)
        st = lib.sla_eig_grad_values(ctypes.byref(cs), 1, v_last.data_ptr(), None, gv.data_ptr(), sh)
        kb.record(stream)
        assert st == 0
        kern_ms.append((ka, kb))
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in kern_ms]
    infos = [r[3] for r in recs]
    inner = sum(i.inner_iters for i in infos)
    tot_s = (sum(eig_ms) + sum(grad_ms)) / 1e3
    tot_s_all, inner_all = aggregate_over_ranks(tot_s, inner, world, dev)
    Bi = b_iter(n, nnz, s_v, s_p, False)
    Bg = b_eig_grad(n, nnz, s_v, s_p)
    peak, peak_kind = measured_peaks()
    achieved = Bi * inner / (sum(eig_ms) / 1e3) / 1e9
    grad_gbs = Bg / (statistics.mean(kern_ms) / 1e3) / 1e9
    th = np.pi / (m + 1)
    mu_exact = 4.0 - 4.0 * np.cos(th)
    out = {
        "metric": EIG_METRIC, "value": inner_all / tot_s_all, "unit": "iters/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean([a + b for a, b in zip(eig_ms, grad_ms)]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (the five-point Laplacian; start vector all ones)",
        "config": {"workload": f"eig_poisson{m}", "n": n, "nnz": nnz, "tol": tol, "inner_factor": 0.01,
                   "step": "smallest eigenpair by inverse iteration + Hellmann-Feynman gradient on the pattern",
                   "l2": "flushed between steps (256 MB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "outer_steps": statistics.mean(i.iters for i in infos), "inner_iters": inner / len(infos),
        "time_to_eigenpair_ms": statistics.mean(eig_ms), "eig_grad_ms": statistics.mean(grad_ms),
        "eig_grad_kernel_ms": statistics.mean(kern_ms),
        "mu": infos[-1].mu, "mu_rel_err_vs_closed_form": abs(infos[-1].mu - mu_exact) / mu_exact,
        "status": sorted({i.status for i in infos}),
        "roofline": {"kernel": "inner CG solves (the engine the solve picks)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                     "bytes_per_iter": Bi, "traffic": None},
        "eig_grad_roofline": {"kernel": "eig_grad_kernel", "bound": "hbm", "achieved": grad_gbs, "peak": peak,
                              "unit": "GB/s", "frac": grad_gbs / peak, "bytes_per_launch": Bg,
                              "timing": "20 launches, each after a 256 MB L2 flush, CUDA events"},
        "gpu_launches": int(launches), "wall_s": wall, "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(config_by_name("poisson1000", m=m), args.cpu_iters)
    return out


BICG_METRIC = ("BiCGStab iters/sec (forward + adjoint) and HBM GB/s (% of roofline), 1M-DOF 2D convection-diffusion "
               "fp64; adjoint ms")


def run_bicgstab(args, rank, world, local_rank):
    """Non-symmetric workload: BiCGStab forward solve and its adjoint (A^T lambda = g by the same solver
    on the partner-permuted values, then grad_values) on the convection-diffusion operator."""
    import torch
    import differentiable_sparse_iterative_gb300 as sla
    from workloads import config_by_name
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = config_by_name(args.config, **({"m": args.grid_m} if args.grid_m else {}))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    A = sla.CSRMatrix.from_numpy(w.A.row_ptr, w.A.col_idx, w.A.values, dev)
    b, g = torch.from_numpy(w.b).to(dev), torch.from_numpy(w.g).to(dev)
    n, nnz = w.A.n, w.A.nnz
    s_v, s_p = 8, w.A.row_ptr.dtype.itemsize
    ws = torch.empty(sla.sla_bicgstab_workspace_bytes(n, nnz, torch.float64), dtype=torch.uint8, device=dev)
    x = torch.empty(n, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    # --loop host: the three-kernel host loop; anything else: the resident kernel
    loop = sla.SLA_LOOP_HOST if args.loop == "host" else sla.SLA_LOOP_AUTO

    def step():
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        _, fi, _ = sla.sla_bicgstab_solve(A, b, rtol=w.rtol, maxit=w.maxit, x=x, workspace=ws, loop=loop)
        e1.record(stream)
        _, _, ai = sla.sla_bicgstab_adjoint(A, x, g, rtol=w.rtol, maxit=w.maxit, workspace=ws, loop=loop)
        e2.record(stream)
        return e0, e1, e2, fi, ai

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = sla.sla_launch_count()
    recs = []
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush_l2(flush)
            recs.append(step())
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    launches = sla.sla_launch_count() - launches0
    fwd_ms = [r[0].elapsed_time(r[1]) for r in recs]
    adj_ms = [r[1].elapsed_time(r[2]) for r in recs]
    iters_f = [r[3].iters for r in recs]
    iters_a = [r[4].iters for r in recs]
    status = {r[3].status for r in recs} | {r[4].status for r in recs}
    tot_s = (sum(fwd_ms) + sum(adj_ms)) / 1e3
    tot_s_all, tot_iters_all = aggregate_over_ranks(tot_s, sum(iters_f) + sum(iters_a), world, dev)
    Bi = b_iter_bicgstab(n, nnz, s_v, s_p)
    peak, peak_kind = measured_peaks()
    fwd_s = sum(fwd_ms) / 1e3
    achieved = Bi * sum(iters_f) / fwd_s / 1e9
    path = recs[-1][3].path
    # the traffic record is the resident kernel's
    tr = None if (args.grid_m or path != "resident") else profiled_traffic(args.config)
    clocks = clk.summary()
    flops_it = flops_iter_bicgstab(n, nnz)
    fp64_peak = fp64_peak_tflops(clocks)
    fp64_ach = flops_it * sum(iters_f) / fwd_s / 1e12
    kernel_name = {"resident": "bi_resident (one persistent cooperative kernel per solve)",
                   "host": "bi_dir_apply + bi_s_apply + bi_update (host loop)"}.get(path, path)
    e2e = None if args.no_e2e else run_e2e(args, w, dev, 0, sla, torch, method="bicgstab")
    out = {
        "metric": BICG_METRIC, "value": tot_iters_all / tot_s_all, "unit": "iters/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean([a + c for a, c in zip(fwd_ms, adj_ms)]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators; no dataset on the pages)",
        "config": {"workload": w.name, "n": n, "nnz": nnz, "rtol": w.rtol, "precond": "none",
                   "step": "forward BiCGStab solve + adjoint (A^T lambda = g by BiCGStab; grad_b, grad_values)",
                   "l2": "flushed between steps (256 MB write); within a solve the iterations reuse L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "loop": args.loop},
        "iters_forward": statistics.mean(iters_f), "iters_adjoint": statistics.mean(iters_a),
        "time_to_tolerance_ms": statistics.mean(fwd_ms), "adjoint_ms": statistics.mean(adj_ms),
        "status": sorted(status), "path": path,
        "fp64": {"achieved_tflops": fp64_ach, "peak_tflops": fp64_peak, "frac": fp64_ach / fp64_peak,
                 "flops_per_iter": flops_it,
                 "peak_basis": "152 SMs x 2 fp64 FMA/clock x 2 flops x max SM clock"},
        "roofline": {"kernel": kernel_name,
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "bytes_per_iter": Bi,
                     "traffic": (tr["dram_bytes_per_iter"] if tr else None),
                     "traffic_unit": "DRAM bytes per BiCGStab iteration (ncu dram__bytes_read + write)",
                     "traffic_source": (tr.get("source") if tr else None)},
        "gpu_launches": int(launches), "wall_s": wall, "clocks": clocks,
    }
    if e2e:
        out["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_iters)
    return out


def run_reference(args, rank, world):
    """The oracle arm: the fp64 CPU oracle timed on the host, on bounded samples of the workload."""
    from workloads import config_by_name
    import oracle
    if rank != 0:
        return None
    # the eigenvalue workload's unit is CG iterations inside the inverse iteration: the oracle's CG
    # on the same matrix is its baseline (a dense eigensolver does not scale to 1M unknowns)
    eig = args.config == "eig_poisson"
    w = config_by_name("poisson1000", m=args.grid_m or 1000) if eig else config_by_name(args.config)
    lib = oracle.load_parallel()
    cores = lib.orc_threads(0)
    g = w.g if w.g is not None else np.random.default_rng(1).standard_normal(w.A.n)
    k = args.ref_iters

    fwd, adj, what = _oracle_pair(w, lib)

    def step():
        f = fwd(k)
        a = adj(f["x"], g, k)
        return f["iters"] + a["iters"]

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    its = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    v = its / dt
    sample = (f"{w.name}: each step at most {k} forward + {k} adjoint {what} iterations (rtol 0; the value counts "
              f"those run) + grad_values, on "
              f"{cores} host cores (the oracle's multi-core build)")
    metric = EIG_METRIC if eig else (BICG_METRIC if what == "BiCGStab" else METRIC)
    return {"impl": "reference", "metric": metric, "value": v, "unit": "iters/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generators)",
            "config": {"workload": w.name, "n": w.A.n, "nnz": w.A.nnz, "rtol": w.rtol},
            "cpu_baseline": {"value": v, "unit": "iters/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "iters/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="poisson1000",
                    help="workload: poisson64, poisson1000 (default), diffusion128_batch64, diffusion4096_jacobi, "
                         "poisson13000_int64 (or config1 .. config5), eig_poisson, convdiff1000_bicgstab")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-iters", type=int, default=0, help="oracle sample size (0: about 15 s of host time)")
    ap.add_argument("--ref-iters", type=int, default=200)
    ap.add_argument("--grid-m", type=int, default=0,
                    help="override the grid side m of the chosen workload (smaller cases for profiling)")
    ap.add_argument("--dist", action="store_true",
                    help="one system split across the ranks (row blocks, halo exchange) instead of replicas")
    ap.add_argument("--loop", choices=["auto", "cluster", "resident", "graph", "host"], default="auto",
                    help="auto (default): resident kernel when the system fits on chip, else graph; "
                         "host: host-driven loop, e.g. for per-kernel ncu")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1 or args.dist:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        if "MASTER_ADDR" not in os.environ:  # a single process without torch.distributed.run
            import socket
            with socket.socket() as sk:
                sk.bind(("127.0.0.1", 0))
                os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(sk.getsockname()[1]), RANK="0",
                                  WORLD_SIZE="1")
        dist.init_process_group("nccl")
    if args.dist:
        out = run_dist(args, rank, world, local_rank)
    elif args.config == "eig_poisson":
        out = run_eig(args, rank, world, local_rank)
    elif args.config == "convdiff1000_bicgstab":
        out = run_bicgstab(args, rank, world, local_rank)
    else:
        out = run_ours(args, rank, world, local_rank)
    if world > 1 or args.dist:
        # before the line is printed: the communicator's teardown may write to stdout, and the
        # JSON line is the last thing on it
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        sys.stdout.flush()
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
