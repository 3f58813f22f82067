"""Distributed row-block CG solve and adjoint over torch.distributed.

Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers and Sparse Tensor
Parallelism for PyTorch" (Chi, Wen), technical summary, Methodology 3 ("distributed layer with
halo exchange"): the matrix is split into contiguous row blocks, one per rank; before its local
SpMV a rank receives the values of the vector at the columns it references but does not own
(its halo); dot products are summed over the ranks.  The CG and its adjoint are those of
Methodology 1-2 (textbook Hestenes-Stiefel CG, optional Jacobi; the adjoint solves A lambda = g
with the same solver, grad_b = lambda, grad_values = -lambda_i x_j on the pattern).

Division of labour:
  * every arithmetic step runs in libsla's kernels (``sla_dist_*`` in ``include/sla.h``): the
    local SpMV with its p.q partial, the x / r / z update with its partials, the direction
    update, the packing of the values a neighbour reads, and the pattern gradient;
  * this module partitions the rows, builds each rank's local block (columns renumbered, halo
    last), plans the exchange, and moves data: halo values by point-to-point send / receive,
    partial sums by all-gather.  Every rank adds the gathered partials in rank order inside the
    kernels, so all ranks hold the same scalars and stop at the same iteration.

On GPUs the process group is NCCL and every tensor stays on the device; with the gloo backend
the exchanged tensors go through host memory (the library's kernels still run on the GPU).

    bounds = partition_rows(row_ptr, world, row_multiple=m)       # whole grid rows
    block = local_block(row_ptr, col_idx, values, bounds, rank)
    solver = DistCG(block, TorchComm(), device="cuda:0")
    x_own, info, hist = solver.solve(b[block.lo:block.hi], rtol=1e-8, maxit=10000)
    grad_b_own, grad_values_local, ainfo = solver.adjoint(x_own, g[block.lo:block.hi], 1e-8, 10000)
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

__all__ = ["partition_rows", "LocalBlock", "local_block", "TorchComm", "LibslaOps", "DistCG", "DistMatVec",
           "dist_matvec"]


# --------------------------------------------------------------------------- partitioning (host)

def partition_rows(row_ptr, world: int, row_multiple: int = 1) -> np.ndarray:
    """Boundaries [world + 1] of contiguous row blocks holding about equal numbers of stored entries.

    Every boundary but the last is a multiple of ``row_multiple`` (for an m x m grid numbered row
    by row, row_multiple = m keeps whole grid rows together, so a rank's halo is one grid row on
    each side).  Blocks may be empty when there are more ranks than units of row_multiple rows.
    """
    rp = np.asarray(row_ptr, dtype=np.int64)
    n = rp.shape[0] - 1
    if world < 1 or row_multiple < 1:
        raise ValueError("world and row_multiple must be >= 1")
    nnz = int(rp[-1])
    bounds = [0]
    for q in range(1, world):
        target = nnz * q / world
        i = int(np.searchsorted(rp, target, side="left"))  # first row starting at or after the target
        i = int(round(i / row_multiple)) * row_multiple
        bounds.append(min(max(i, bounds[-1]), n))
    bounds.append(n)
    return np.asarray(bounds, dtype=np.int64)


@dataclass
class LocalBlock:
    """One rank's rows [lo, hi) with columns renumbered: owned columns 0..n_own-1, then the halo.

    row_ptr / col_idx / values describe the square CSR of order n_ext whose rows n_own.. are empty
    (the form libsla's distributed calls take).  recv[peer] = (start, count): the halo slots
    n_own + start .. n_own + start + count - 1 hold peer's values (the halo is sorted by global
    column, and each peer owns a contiguous range, so its columns are contiguous).  send[peer]:
    local indices of the owned values peer reads, in the order peer stores them (set by plan_exchange).
    """
    rank: int
    world: int
    lo: int
    hi: int
    bounds: np.ndarray
    row_ptr: np.ndarray
    col_idx: np.ndarray
    values: np.ndarray
    halo_global: np.ndarray
    recv: Dict[int, Tuple[int, int]]
    send: Dict[int, np.ndarray] = field(default_factory=dict)
    # the local block's transpose (square of order n_ext: row j lists the owned rows i with a stored
    # (i, j)), for the backward of a distributed product; its values are values[t_perm]
    t_row_ptr: Optional[np.ndarray] = None
    t_col_idx: Optional[np.ndarray] = None
    t_perm: Optional[np.ndarray] = None

    @property
    def n_own(self) -> int:
        return self.hi - self.lo

    @property
    def n_ext(self) -> int:
        return self.n_own + int(self.halo_global.shape[0])

    @property
    def nnz(self) -> int:
        return int(self.col_idx.shape[0])


def local_block(row_ptr, col_idx, values, bounds, rank: int) -> LocalBlock:
    """The local block of `rank` from the global CSR (host arrays) and the partition `bounds`."""
    rp = np.asarray(row_ptr, dtype=np.int64)
    ci = np.asarray(col_idx)
    bounds = np.asarray(bounds, dtype=np.int64)
    world = bounds.shape[0] - 1
    lo, hi = int(bounds[rank]), int(bounds[rank + 1])
    e0, e1 = int(rp[lo]), int(rp[hi])
    cols = ci[e0:e1].astype(np.int64)
    own = (cols >= lo) & (cols < hi)
    halo = np.unique(cols[~own])
    loc = np.empty(cols.shape[0], dtype=np.int64)
    loc[own] = cols[own] - lo
    loc[~own] = (hi - lo) + np.searchsorted(halo, cols[~own])
    n_own = hi - lo
    rp_loc = np.concatenate([rp[lo:hi + 1] - e0, np.full(halo.shape[0], e1 - e0, dtype=np.int64)])
    rp_loc = rp_loc.astype(np.asarray(row_ptr).dtype)
    owner = np.searchsorted(bounds, halo, side="right") - 1
    recv: Dict[int, Tuple[int, int]] = {}
    for peer in np.unique(owner):
        idx = np.nonzero(owner == peer)[0]
        recv[int(peer)] = (int(idx[0]), int(idx.shape[0]))
    # transpose of the local block: entries sorted by column, stably (so by row within a column)
    n_ext = n_own + halo.shape[0]
    rows = np.repeat(np.arange(n_own, dtype=np.int64), np.diff(rp[lo:hi + 1]))
    t_perm = np.argsort(loc, kind="stable").astype(np.int64)
    t_rp = np.concatenate([[0], np.cumsum(np.bincount(loc, minlength=n_ext))]).astype(rp_loc.dtype)
    return LocalBlock(rank, world, lo, hi, bounds, rp_loc, loc.astype(np.int32),
                      np.ascontiguousarray(np.asarray(values)[e0:e1]), halo, recv,
                      t_row_ptr=t_rp, t_col_idx=rows[t_perm].astype(np.int32), t_perm=t_perm)


def plan_exchange(block: LocalBlock, comm) -> None:
    """Fills block.send: every rank tells each owner which of its columns it reads."""
    wants = {peer: block.halo_global[start:start + count].tolist() for peer, (start, count) in block.recv.items()}
    everyone = comm.all_gather_object(wants)
    send = {}
    for peer in range(block.world):
        cols = everyone[peer].get(block.rank)
        if cols:
            send[peer] = np.asarray(cols, dtype=np.int64) - block.lo
    block.send = send


# --------------------------------------------------------------------------- communication

class TorchComm:
    """Halo exchange and partial-sum gathering over a torch.distributed process group.

    NCCL: device tensors are sent and gathered in place.  gloo: through host copies."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.host = dist.get_backend(group) != "nccl"

    def all_gather_object(self, obj) -> list:
        out = [None] * self.world
        self.dist.all_gather_object(out, obj, group=self.group)
        return out

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        """Every rank's copy of t, concatenated in rank order (on t's device)."""
        if self.host:
            src = t.cpu()
            parts = [torch.empty_like(src) for _ in range(self.world)]
            self.dist.all_gather(parts, src, group=self.group)
            return torch.cat(parts).to(t.device)
        out = torch.empty(self.world * t.numel(), dtype=t.dtype, device=t.device)
        self.dist.all_gather_into_tensor(out, t.contiguous(), group=self.group)
        return out

    def exchange(self, sends: Dict[int, torch.Tensor], recvs: Dict[int, torch.Tensor]) -> None:
        """Sends sends[peer] to peer and receives into recvs[peer] (views are filled in place)."""
        dist = self.dist
        if not sends and not recvs:
            return
        if self.host:
            hs = {p: t.cpu() for p, t in sends.items()}
            hr = {p: torch.empty(t.shape, dtype=t.dtype) for p, t in recvs.items()}
        else:
            hs, hr = sends, recvs
        ops = [dist.P2POp(dist.isend, t, p, group=self.group) for p, t in sorted(hs.items())]
        ops += [dist.P2POp(dist.irecv, t, p, group=self.group) for p, t in sorted(hr.items())]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        if self.host:
            for p, t in recvs.items():
                t.copy_(hr[p])


# --------------------------------------------------------------------------- local steps (libsla)

class LibslaOps:
    """One rank's steps of the distributed CG, each a libsla kernel on the rank's GPU."""

    def __init__(self):
        from . import lib
        self.lib = lib()

    @staticmethod
    def _p(t: Optional[torch.Tensor]):
        from . import _dev_ptr
        return _dev_ptr(t)  # CUDA tensors only: there is no CPU path

    def _check(self, st: int, where: str):
        from . import SlaError
        if st != 0:
            raise SlaError(st, where)

    def state(self, device) -> torch.Tensor:
        nbytes = int(self.lib.sla_dist_state_bytes())
        return torch.empty(nbytes // 8, dtype=torch.float64, device=device)

    def begin(self, A, n_own, b, opts, x, r, z, p_ext, dinv, part5, state, stream):
        from . import _csr_struct
        self._check(self.lib.sla_dist_cg_begin(ctypes.byref(_csr_struct(A)), n_own, self._p(b), ctypes.byref(opts),
                                               self._p(x), self._p(r), self._p(z), self._p(p_ext), self._p(dinv),
                                               self._p(part5), self._p(state), stream), "sla_dist_cg_begin")

    def start(self, gathered, ranks, state, history, stream):
        self._check(self.lib.sla_dist_cg_start(self._p(gathered), ranks, self._p(state), self._p(history), stream),
                    "sla_dist_cg_start")

    def spmv(self, A, n_own, p_ext, q, part1, state, stream):
        from . import _csr_struct
        self._check(self.lib.sla_dist_cg_spmv(ctypes.byref(_csr_struct(A)), n_own, self._p(p_ext), self._p(q),
                                              self._p(part1), self._p(state), stream), "sla_dist_cg_spmv")

    def update(self, n_own, dtype, precond, gathered, ranks, x, r, p_ext, q, dinv, z, part2, state, stream):
        self._check(self.lib.sla_dist_cg_update(n_own, dtype, precond, self._p(gathered), ranks, self._p(x),
                                                self._p(r), self._p(p_ext), self._p(q), self._p(dinv), self._p(z),
                                                self._p(part2), self._p(state), stream), "sla_dist_cg_update")

    def direction(self, n_own, dtype, gathered, ranks, zr, p_ext, history, state, stream):
        self._check(self.lib.sla_dist_cg_direction(n_own, dtype, self._p(gathered), ranks, self._p(zr),
                                                   self._p(p_ext), self._p(history), self._p(state), stream),
                    "sla_dist_cg_direction")

    def pack(self, n, dtype, v, idx, buf, stream):
        self._check(self.lib.sla_dist_pack(n, dtype, self._p(v), self._p(idx), int(idx.numel()), self._p(buf), stream),
                    "sla_dist_pack")

    def info(self, state, stream):
        from . import _abi
        ci = _abi.sla_cg_info()
        done = ctypes.c_int32(0)
        self._check(self.lib.sla_dist_cg_info(self._p(state), ctypes.byref(ci), ctypes.byref(done), stream),
                    "sla_dist_cg_info")
        return ci, int(done.value)

    def product(self, A, x, y, stream):
        from . import _csr_struct
        self._check(self.lib.sla_spmv(ctypes.byref(_csr_struct(A)), self._p(x), self._p(y), stream), "sla_spmv")

    def scatter_add(self, n, dtype, v, idx, buf, stream):
        self._check(self.lib.sla_dist_scatter_add(n, dtype, self._p(v), self._p(idx), int(idx.numel()), self._p(buf),
                                                  stream), "sla_dist_scatter_add")

    def matvec_grad(self, A, gy, x, gv, stream):
        from . import _csr_struct
        self._check(self.lib.sla_matvec_grad_values(ctypes.byref(_csr_struct(A)), self._p(gy), self._p(x),
                                                    self._p(gv), stream), "sla_matvec_grad_values")

    def grad_values(self, A, lam_ext, x_ext, gv, stream):
        from . import _csr_struct
        self._check(self.lib.sla_grad_values(ctypes.byref(_csr_struct(A)), self._p(lam_ext), self._p(x_ext),
                                             self._p(gv), stream), "sla_grad_values")


# --------------------------------------------------------------------------- the solver

class DistCG:
    """Distributed CG and adjoint for one rank's LocalBlock.

    ops: the local steps (LibslaOps: libsla kernels on `device`).  comm: TorchComm (or any object
    with rank, world, all_gather, all_gather_object and exchange).  The exchange plan is made
    collectively when the solver is built, so every rank must build its DistCG together.
    """

    def __init__(self, block: LocalBlock, comm, device="cuda", ops=None):
        from . import CSRMatrix
        self.block = block
        self.comm = comm
        self.device = torch.device(device)
        self.ops = ops if ops is not None else LibslaOps()
        if not block.send and block.world > 1:
            plan_exchange(block, comm)
        dev = self.device
        self.A = CSRMatrix(torch.from_numpy(np.ascontiguousarray(block.row_ptr)).to(dev),
                           torch.from_numpy(np.ascontiguousarray(block.col_idx)).to(dev),
                           torch.from_numpy(np.ascontiguousarray(block.values)).to(dev))
        self.vdtype = self.A.values.dtype
        self.t_row_ptr = torch.from_numpy(np.ascontiguousarray(block.t_row_ptr)).to(dev)
        self.t_col_idx = torch.from_numpy(np.ascontiguousarray(block.t_col_idx)).to(dev)
        self.t_perm = torch.from_numpy(np.ascontiguousarray(block.t_perm)).to(dev)
        self.send_idx = {p: torch.from_numpy(idx).to(dev) for p, idx in block.send.items()}
        self.send_buf = {p: torch.empty(idx.shape[0], dtype=self.vdtype, device=dev)
                         for p, idx in block.send.items()}
        self.state = self.ops.state(dev)

    def _stream(self) -> int:
        if self.device.type == "cuda":
            return torch.cuda.current_stream(self.device).cuda_stream
        return 0

    def _dtype_code(self) -> int:
        return 1 if self.vdtype == torch.float64 else 0

    def exchange(self, v_ext: torch.Tensor) -> None:
        """Fills the halo part of v_ext (n_ext entries) with the owners' values."""
        st = self._stream()
        n_own = self.block.n_own
        for p, idx in self.send_idx.items():
            self.ops.pack(n_own, self._dtype_code(), v_ext, idx, self.send_buf[p], st)
        recvs = {p: v_ext[n_own + s:n_own + s + c] for p, (s, c) in self.block.recv.items()}
        self.comm.exchange(self.send_buf, recvs)

    def solve(self, b_own: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000, precond: int = 0,
              history: bool = False, unroll: int = 8):
        """Solves the distributed system; returns (x_ext, info, history or None).

        x_ext has n_ext entries: the owned solution first (x_ext[:n_own]); its halo part is
        scratch.  info is libsla's sla_cg_info (iterations, relative residual, status)."""
        from . import _opts
        blk, ops, dev = self.block, self.ops, self.device
        n_own, n_ext, R = blk.n_own, blk.n_ext, self.comm.world
        vd = self.vdtype
        jac = precond == 1
        x = torch.zeros(n_ext, dtype=vd, device=dev)
        r = torch.empty(max(n_own, 1), dtype=vd, device=dev)
        q = torch.empty(max(n_own, 1), dtype=vd, device=dev)
        p = torch.zeros(n_ext, dtype=vd, device=dev)
        z = torch.empty(max(n_own, 1), dtype=vd, device=dev) if jac else None
        dinv = torch.empty(max(n_own, 1), dtype=vd, device=dev) if jac else None
        part5 = torch.zeros(5, dtype=torch.float64, device=dev)
        part1 = torch.zeros(1, dtype=torch.float64, device=dev)
        part2 = torch.zeros(2, dtype=torch.float64, device=dev)
        hist = torch.full((maxit + 1,), float("nan"), dtype=torch.float64, device=dev) if history else None
        b = b_own.to(device=dev, dtype=vd).contiguous()
        st = self._stream()
        code = self._dtype_code()
        ops.begin(self.A, n_own, b, _opts(rtol, maxit, precond), x, r, z, p, dinv, part5, self.state, st)
        ops.start(self.comm.all_gather(part5), R, self.state, hist, st)
        info, done = ops.info(self.state, st)
        k = 0
        while not done and k < maxit:
            self.exchange(p)
            for u in range(unroll):
                ops.spmv(self.A, n_own, p, q, part1, self.state, st)
                g1 = self.comm.all_gather(part1)
                ops.update(n_own, code, precond, g1, R, x, r, p, q, dinv, z, part2, self.state, st)
                g2 = self.comm.all_gather(part2)
                ops.direction(n_own, code, g2, R, z if jac else r, p, hist, self.state, st)
                if u + 1 < unroll:
                    self.exchange(p)
            k += unroll
            info, done = ops.info(self.state, st)
        if hist is not None:
            hist = hist[: info.iters + 1]
        return x, info, hist

    # ------------------------------------------------------------------ distributed product

    def matvec(self, x_own: torch.Tensor, values: Optional[torch.Tensor] = None):
        """y = A x for this rank's rows: the halo of x is exchanged first (forward halo exchange).
        Returns (y_own, x_ext); values (optional) replaces the local block's values."""
        from . import CSRMatrix
        blk = self.block
        A = self.A if values is None else CSRMatrix(self.A.row_ptr, self.A.col_idx, values)
        xe = torch.zeros(blk.n_ext, dtype=self.vdtype, device=self.device)
        xe[: blk.n_own] = x_own.to(device=self.device, dtype=self.vdtype)
        self.exchange(xe)
        y = torch.empty(blk.n_ext, dtype=self.vdtype, device=self.device)
        self.ops.product(A, xe, y, self._stream())
        return y[: blk.n_own], xe

    def matvec_backward(self, gy_own: torch.Tensor, x_ext: torch.Tensor, values: Optional[torch.Tensor] = None):
        """Backward of y = A x for this rank's rows (Methodology 3's transposed halo exchange).

        The rank forms A_loc^T gy over every column its rows touch; the halo part belongs to the
        neighbours and is sent to them, and the contributions they computed for this rank's owned
        entries are received and added in (rank order).  Returns (grad_x_own, grad_values_local)
        with grad_values[e] = gy_i x_j on the rank's entries."""
        from . import CSRMatrix
        blk, ops, st, code = self.block, self.ops, self._stream(), self._dtype_code()
        vals = self.A.values if values is None else values
        A = CSRMatrix(self.A.row_ptr, self.A.col_idx, vals)
        gye = torch.zeros(blk.n_ext, dtype=self.vdtype, device=self.device)
        gye[: blk.n_own] = gy_own.to(device=self.device, dtype=self.vdtype)
        vt = torch.empty(blk.nnz, dtype=self.vdtype, device=self.device)
        if blk.nnz:
            ops.pack(blk.nnz, code, vals, self.t_perm, vt, st)  # values in the transpose's order
        At = CSRMatrix(self.t_row_ptr, self.t_col_idx, vt)
        gxe = torch.empty(blk.n_ext, dtype=self.vdtype, device=self.device)
        ops.product(At, gye, gxe, st)
        sends = {p: gxe[blk.n_own + s:blk.n_own + s + c] for p, (s, c) in blk.recv.items()}
        recvs = {p: torch.empty(idx.numel(), dtype=self.vdtype, device=self.device)
                 for p, idx in self.send_idx.items()}
        self.comm.exchange(sends, recvs)
        gx = gxe[: blk.n_own]
        for p in sorted(recvs):
            ops.scatter_add(blk.n_own, code, gx, self.send_idx[p], recvs[p], st)
        gv = torch.empty(blk.nnz, dtype=self.vdtype, device=self.device)
        if blk.nnz:
            ops.matvec_grad(A, gye, x_ext, gv, st)
        return gx, gv

    def adjoint(self, x: torch.Tensor, g_own: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000,
                precond: int = 0, unroll: int = 8):
        """Adjoint of x = A^{-1} b (Methodology 2) for this rank's rows.

        x: the forward solution, owned part first (n_own or n_ext entries).  Solves A lambda = g
        distributed (A symmetric), then fills the halo of a copy of x and forms
        grad_values = -lambda_i x_j on the local pattern (the rank's stored entries, in the global
        CSR order of its rows).  Returns (grad_b_own = lambda_own, grad_values_local, info)."""
        lam, info, _ = self.solve(g_own, rtol, maxit, precond, False, unroll)
        xe = torch.zeros(self.block.n_ext, dtype=self.vdtype, device=self.device)
        xe[: self.block.n_own] = x[: self.block.n_own].to(device=self.device, dtype=self.vdtype)
        self.exchange(xe)
        gv = torch.empty(self.block.nnz, dtype=self.vdtype, device=self.device)
        if self.block.nnz:
            self.ops.grad_values(self.A, lam, xe, gv, self._stream())
        return lam[: self.block.n_own], gv, info


class DistMatVec(torch.autograd.Function):
    """Differentiable distributed y = A x for one rank's rows (forward halo exchange; transposed
    halo exchange in backward).  Gradients flow to the rank's stored values and owned x."""

    @staticmethod
    def forward(ctx, values, x_own, solver):
        y, xe = solver.matvec(x_own, values)
        ctx.solver = solver
        ctx.save_for_backward(values, xe)
        return y.clone()

    @staticmethod
    def backward(ctx, gy):
        values, xe = ctx.saved_tensors
        gx, gv = ctx.solver.matvec_backward(gy.contiguous(), xe, values)
        return gv, gx, None


def dist_matvec(solver: DistCG, values: torch.Tensor, x_own: torch.Tensor) -> torch.Tensor:
    """y_own = (A x)_own, differentiable with respect to the rank's values and owned x."""
    return DistMatVec.apply(values, x_own, solver)
