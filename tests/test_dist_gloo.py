"""Distributed row-block CG and adjoint on gloo CPU ranks (world sizes 2 and 3), against the oracle.

The distributed layer (differentiable_sparse_iterative_gb300.distributed, after the torch-sla
summary's Methodology 3: row blocks, halo exchange before the local SpMV, dot products summed
over ranks) runs over real torch.distributed process groups on CPU.  The local steps are the numpy
stand-in of tests/dist_numpy_ops.py (the product runs them as libsla kernels; the GPU test of
that path is tests/test_gpu_dist.py).  Checked on rank 0 against the single-process fp64 oracle:
the solution at 1e-9, the first 50 residual-history entries at 1e-8, grad_b and grad_values at
1e-7, and the iteration counts.  Also the partition and local blocks on their own.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))

from differentiable_sparse_iterative_gb300 import distributed as D  # noqa: E402
import oracle  # noqa: E402
from workloads import poisson_5pt, diffusion_dirichlet, random_spd  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rel(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def _case(name):
    if name == "poisson":
        m = 30
        A = poisson_5pt(m)
        return A, m, 0
    if name == "diffusion_jacobi":
        m = 24
        A = diffusion_dirichlet(m, np.random.default_rng(3).lognormal(0, 1.0, 2 * m * (m + 1)))
        return A, m, 1
    if name == "tiny":  # a 2 x 2 grid on more ranks than it has grid rows: one rank owns nothing
        return poisson_5pt(2), 2, 0
    A = random_spd(700, 5.0, 4, long_rows=2)
    return A, 1, 0


# --------------------------------------------------------------------------- host logic alone

@pytest.mark.parametrize("world", [1, 2, 3, 5])
@pytest.mark.parametrize("name", ["poisson", "random"])
def test_partition_and_local_blocks_reproduce_the_global_product(name, world):
    sp = pytest.importorskip("scipy.sparse")
    A, mult, _ = _case(name)
    bounds = D.partition_rows(A.row_ptr, world, mult)
    assert bounds[0] == 0 and bounds[-1] == A.n and np.all(np.diff(bounds) >= 0)
    assert np.all(bounds[1:-1] % mult == 0)
    S = sp.csr_matrix((A.values, A.col_idx, A.row_ptr.astype(np.int64)), shape=(A.n, A.n))
    x = np.random.default_rng(5).standard_normal(A.n)
    y = S @ x
    blocks = [D.local_block(A.row_ptr, A.col_idx, A.values, bounds, r) for r in range(world)]
    total_nnz = 0
    for blk in blocks:
        # the local block of order n_ext, its halo filled from the global vector
        xe = np.concatenate([x[blk.lo:blk.hi], x[blk.halo_global]])
        L = sp.csr_matrix((blk.values, blk.col_idx, blk.row_ptr.astype(np.int64)), shape=(blk.n_ext, blk.n_ext))
        ye = L @ xe
        assert np.array_equal(ye[: blk.n_own], y[blk.lo:blk.hi]) or _rel(ye[: blk.n_own], y[blk.lo:blk.hi]) < 1e-15
        assert not ye[blk.n_own:].any()  # halo rows are empty
        assert np.all((blk.halo_global < blk.lo) | (blk.halo_global >= blk.hi))
        total_nnz += blk.nnz
        # the receive segments cover the halo, peer by peer, in order
        covered = 0
        for peer, (s, c) in sorted(blk.recv.items()):
            assert s == covered and peer != blk.rank
            own = blk.halo_global[s:s + c]
            assert np.all((own >= bounds[peer]) & (own < bounds[peer + 1]))
            covered += c
        assert covered == blk.halo_global.shape[0]
    assert total_nnz == A.nnz


def test_grid_partition_keeps_whole_grid_rows():
    m = 40
    A = poisson_5pt(m)
    bounds = D.partition_rows(A.row_ptr, 3, m)
    blk = D.local_block(A.row_ptr, A.col_idx, A.values, bounds, 1)
    # a middle rank reads one grid row from each neighbour
    assert sorted(blk.recv) == [0, 2] and blk.recv[0][1] == m and blk.recv[2][1] == m


# --------------------------------------------------------------------------- gloo ranks

def _rank_main(rank, world, port, name, out_dir):
    sys.path[:0] = [ROOT, TESTS]
    import torch.distributed as dist
    from dist_numpy_ops import NumpyOps
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, mult, precond = _case(name)
        rng = np.random.default_rng(11)
        b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
        bounds = D.partition_rows(A.row_ptr, world, mult)
        blk = D.local_block(A.row_ptr, A.col_idx, A.values, bounds, rank)
        solver = D.DistCG(blk, D.TorchComm(), device="cpu", ops=NumpyOps())
        x, info, hist = solver.solve(torch.from_numpy(b[blk.lo:blk.hi].copy()), rtol=1e-10, maxit=2000,
                                     precond=precond, history=True, unroll=3)
        gb, gv, ainfo = solver.adjoint(x, torch.from_numpy(g[blk.lo:blk.hi].copy()), rtol=1e-10, maxit=2000,
                                       precond=precond, unroll=3)
        mine = (blk.lo, blk.hi, x[: blk.n_own].numpy().copy(), gb.numpy().copy(), gv.numpy().copy(),
                info.iters, info.status, ainfo.iters, ainfo.status, hist.numpy().copy())
        everyone = solver.comm.all_gather_object(mine)
        if rank == 0:
            xs = np.concatenate([e[2] for e in everyone])
            gbs = np.concatenate([e[3] for e in everyone])
            gvs = np.concatenate([e[4] for e in everyone])
            np.savez(os.path.join(out_dir, f"{name}_{world}.npz"), x=xs, gb=gbs, gv=gvs,
                     iters=[e[5] for e in everyone], status=[e[6] for e in everyone],
                     aiters=[e[7] for e in everyone], astatus=[e[8] for e in everyone], hist=everyone[0][9],
                     hists_equal=all(np.array_equal(e[9], everyone[0][9]) for e in everyone))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,name", [(2, "poisson"), (3, "poisson"), (2, "diffusion_jacobi"),
                                        (3, "diffusion_jacobi"), (2, "random"), (3, "random"), (3, "tiny")])
def test_distributed_cg_and_adjoint_match_the_oracle(name, world, tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(world, _free_port(), name, str(tmp_path)), nprocs=world, join=True)
    res = np.load(tmp_path / f"{name}_{world}.npz")
    A, _, precond = _case(name)
    rng = np.random.default_rng(11)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=2000, precond=precond, history=True)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-10, maxit=2000, precond=precond)
    # every rank stopped at the same iteration with the same status and history
    assert len(set(res["iters"])) == 1 and len(set(res["status"])) == 1 and bool(res["hists_equal"])
    assert res["status"][0] == ref["status"] == 0 and res["astatus"][0] == adj["status"] == 0
    assert abs(int(res["iters"][0]) - ref["iters"]) <= 1 and abs(int(res["aiters"][0]) - adj["iters"]) <= 1
    assert _rel(res["x"], ref["x"]) <= 1e-9
    # residual histories over the first 50 iterations, or up to the horizon where the oracle's own
    # trajectory departs under one-ulp changes of b (rounding-order sensitivity of CG on small
    # irregular matrices; see gpu_helpers.rounding_sensitivity)
    from gpu_helpers import rounding_sensitivity, check_history
    horizon, _ = rounding_sensitivity(A, b, precond, 1e-10, 2000)
    check_history(res["hist"], ref["history"], k=min(50, horizon - 1))
    assert horizon >= 8 or name in ("random", "tiny")
    assert _rel(res["gb"], adj["grad_b"]) <= 1e-7
    assert res["gv"].shape == (A.nnz,)  # the ranks' entries, in global CSR order
    assert _rel(res["gv"], adj["grad_values"]) <= 1e-7


# --------------------------------------------------------------------------- distributed product

def _nonsym_csr(n, per_row, seed):
    """A structurally non-symmetric random CSR matrix with a stored diagonal."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(n):
        c = set(rng.choice(n, int(rng.integers(0, per_row + 1)), replace=False).tolist()) | {i}
        rows.append(np.array(sorted(c), dtype=np.int32))
    rp = np.concatenate([[0], np.cumsum([r.shape[0] for r in rows])]).astype(np.int32)
    return rp, np.concatenate(rows), rng.standard_normal(int(rp[-1]))


def _matvec_rank(rank, world, port, out_dir):
    sys.path[:0] = [ROOT, TESTS]
    import torch.distributed as dist
    from dist_numpy_ops import NumpyOps
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rp, ci, v = _nonsym_csr(400, 6, 21)
        rng = np.random.default_rng(22)
        x, gy = rng.standard_normal(400), rng.standard_normal(400)
        bounds = D.partition_rows(rp, world, 1)
        blk = D.local_block(rp, ci, v, bounds, rank)
        solver = D.DistCG(blk, D.TorchComm(), device="cpu", ops=NumpyOps())
        vals = torch.from_numpy(blk.values.copy()).requires_grad_(True)
        xo = torch.from_numpy(x[blk.lo:blk.hi].copy()).requires_grad_(True)
        y = D.dist_matvec(solver, vals, xo)
        y.backward(torch.from_numpy(gy[blk.lo:blk.hi].copy()))
        mine = (y.detach().numpy().copy(), xo.grad.numpy().copy(), vals.grad.numpy().copy())
        everyone = solver.comm.all_gather_object(mine)
        if rank == 0:
            np.savez(os.path.join(out_dir, f"mv_{world}.npz"), y=np.concatenate([e[0] for e in everyone]),
                     gx=np.concatenate([e[1] for e in everyone]), gv=np.concatenate([e[2] for e in everyone]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_distributed_matvec_and_transposed_exchange(world, tmp_path):
    # a structurally non-symmetric matrix: grad_x = A^T gy needs the contributions other ranks
    # computed for this rank's entries (the transposed halo exchange)
    import torch.multiprocessing as mp
    mp.spawn(_matvec_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = np.load(tmp_path / f"mv_{world}.npz")
    rp, ci, v = _nonsym_csr(400, 6, 21)
    rng = np.random.default_rng(22)
    x, gy = rng.standard_normal(400), rng.standard_normal(400)
    assert _rel(res["y"], oracle.spmv(rp, ci, v, x)) <= 1e-14
    assert _rel(res["gx"], oracle.spmv_transpose(rp, ci, v, gy)) <= 1e-14
    assert np.array_equal(res["gv"], oracle.matvec_grad_values(rp, ci, gy, x))
