"""The distributed row-block CG and adjoint with libsla's kernels on the GPU, against the oracle.

Each rank is a spawned process using cuda:0 (one GPU is available to the tests), with a gloo
process group: halo values and partial sums travel through host memory, so no kernel of one rank
waits on another rank's kernels.  The local steps are libsla's sla_dist_* kernels and
sla_grad_values (LibslaOps), as on a multi-GPU NCCL run.  Checked on rank 0 against the
single-process fp64 oracle at the fp64 bars (solution 1e-9, history 1e-8 over 50 iterations,
grad_b and grad_values 1e-7).
"""
import os
import socket
import sys

import numpy as np
import pytest

from gpu_helpers import oracle, torch, check_history, rel  # noqa: F401

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(name):
    from workloads import poisson_5pt, diffusion_dirichlet
    if name == "poisson":
        m = 120
        return poisson_5pt(m), m, 0, np.float64
    if name == "poisson_int64":
        m = 90
        return poisson_5pt(m, rowptr64=True), m, 0, np.float64
    if name == "tiny":  # a 2 x 2 grid on three ranks: the last one owns no rows
        return poisson_5pt(2), 2, 0, np.float64
    m = 100
    A = diffusion_dirichlet(m, np.random.default_rng(3).lognormal(0, 1.0, 2 * m * (m + 1)))
    return A, m, 1, np.float64


def _rank_main(rank, world, port, name, out_dir):
    sys.path[:0] = [ROOT, TESTS]
    import torch.distributed as dist
    from differentiable_sparse_iterative_gb300 import distributed as D
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, mult, precond, dt = _case(name)
        rng = np.random.default_rng(21)
        b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
        bounds = D.partition_rows(A.row_ptr, world, mult)
        blk = D.local_block(A.row_ptr, A.col_idx, A.values.astype(dt), bounds, rank)
        solver = D.DistCG(blk, D.TorchComm(), device="cuda:0")
        x, info, hist = solver.solve(torch.from_numpy(b[blk.lo:blk.hi].copy()), rtol=1e-10, maxit=5000,
                                     precond=precond, history=True)
        gb, gv, ainfo = solver.adjoint(x, torch.from_numpy(g[blk.lo:blk.hi].copy()), rtol=1e-10, maxit=5000,
                                       precond=precond)
        torch.cuda.synchronize()
        mine = (x[: blk.n_own].cpu().numpy(), gb.cpu().numpy(), gv.cpu().numpy(), info.iters, info.status,
                ainfo.iters, ainfo.status, hist.cpu().numpy())
        everyone = solver.comm.all_gather_object(mine)
        if rank == 0:
            np.savez(os.path.join(out_dir, "res.npz"), x=np.concatenate([e[0] for e in everyone]),
                     gb=np.concatenate([e[1] for e in everyone]), gv=np.concatenate([e[2] for e in everyone]),
                     iters=[e[3] for e in everyone], status=[e[4] for e in everyone],
                     aiters=[e[5] for e in everyone], astatus=[e[6] for e in everyone], hist=everyone[0][7],
                     hists_equal=all(np.array_equal(e[7], everyone[0][7]) for e in everyone))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,name", [(1, "poisson"), (2, "poisson"), (3, "poisson_int64"), (2, "diffusion_jacobi"),
                                        (3, "tiny")])
def test_distributed_cg_and_adjoint_on_gpu(world, name, tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(world, _free_port(), name, str(tmp_path)), nprocs=world, join=True)
    res = np.load(tmp_path / "res.npz")
    A, _, precond, _ = _case(name)
    rng = np.random.default_rng(21)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=5000, precond=precond, history=True)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-10, maxit=5000, precond=precond)
    assert len(set(res["iters"])) == 1 and len(set(res["status"])) == 1 and bool(res["hists_equal"])
    assert res["status"][0] == ref["status"] == 0 and res["astatus"][0] == adj["status"] == 0
    assert abs(int(res["iters"][0]) - ref["iters"]) <= 1 and abs(int(res["aiters"][0]) - adj["iters"]) <= 1
    assert rel(res["x"], ref["x"]) <= 1e-9
    check_history(res["hist"], ref["history"], k=min(50, len(ref["history"]) - 1))
    assert rel(res["gb"], adj["grad_b"]) <= 1e-7
    assert res["gv"].shape == (A.nnz,)
    assert rel(res["gv"], adj["grad_values"]) <= 1e-7


def _matvec_rank(rank, world, port, out_dir):
    sys.path[:0] = [ROOT, TESTS]
    import torch.distributed as dist
    from differentiable_sparse_iterative_gb300 import distributed as D
    from test_dist_gloo import _nonsym_csr
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rp, ci, v = _nonsym_csr(3000, 6, 31)
        rng = np.random.default_rng(32)
        x, gy = rng.standard_normal(3000), rng.standard_normal(3000)
        bounds = D.partition_rows(rp, world, 1)
        blk = D.local_block(rp, ci, v, bounds, rank)
        solver = D.DistCG(blk, D.TorchComm(), device="cuda:0")
        vals = torch.from_numpy(blk.values.copy()).cuda().requires_grad_(True)
        xo = torch.from_numpy(x[blk.lo:blk.hi].copy()).cuda().requires_grad_(True)
        y = D.dist_matvec(solver, vals, xo)
        y.backward(torch.from_numpy(gy[blk.lo:blk.hi].copy()).cuda())
        torch.cuda.synchronize()
        mine = (y.detach().cpu().numpy(), xo.grad.cpu().numpy(), vals.grad.cpu().numpy())
        everyone = solver.comm.all_gather_object(mine)
        if rank == 0:
            np.savez(os.path.join(out_dir, "mv.npz"), y=np.concatenate([e[0] for e in everyone]),
                     gx=np.concatenate([e[1] for e in everyone]), gv=np.concatenate([e[2] for e in everyone]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [1, 2, 3])
def test_distributed_matvec_transposed_exchange_on_gpu(world, tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_matvec_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = np.load(tmp_path / "mv.npz")
    from test_dist_gloo import _nonsym_csr
    rp, ci, v = _nonsym_csr(3000, 6, 31)
    rng = np.random.default_rng(32)
    x, gy = rng.standard_normal(3000), rng.standard_normal(3000)
    assert rel(res["y"], oracle.spmv(rp, ci, v, x)) <= 1e-14
    assert rel(res["gx"], oracle.spmv_transpose(rp, ci, v, gy)) <= 1e-14
    assert np.array_equal(res["gv"], oracle.matvec_grad_values(rp, ci, gy, x))
