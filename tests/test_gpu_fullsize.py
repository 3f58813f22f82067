"""Full-size workloads through the C ABI, in the launch configuration the benchmark times,
compared element by element with the oracle.

The two large systems use the oracle's multi-core build (same arithmetic as the plain build;
dot products summed in fixed chunks, so its results do not depend on the thread count):
config 2 (1M-DOF Poisson, fp64, rtol 1e-8), config 4 (16.8M-DOF variable-coefficient
diffusion, Jacobi PCG, rtol 1e-8) and config 5 (169M-DOF Poisson, int64 row_ptr, 1000 fixed
iterations) each compare the solution (1e-9), the first 50 residual-history entries (1e-8) and
the adjoint gradients grad_b and grad_values (1e-7), the oracle's adjoint chaining from its own
forward solution.  A fourth case crosses the 32-bit entry-offset boundary: a banded SPD
pattern with 2.18e9 stored entries and int64 row_ptr, five iterations forward and adjoint against
the oracle, grad_values on sampled rows past entry 2^31.  Wall time on the GPU machine's host cores is
dominated by the oracle: see the timing printed with -s.
"""
import time

import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, to_dev, t, check_history, X_TOL_F64, GRAD_TOL_F64, ITER_SLACK_F64
from workloads import config2, config4, config5

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _free_host_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable"):
                    return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


def test_config2_full_oracle():
    w = config2()
    dA = to_dev(w.A)
    b, g = t(w.b), t(w.g)
    x, info, hist = sla.sla_cg_solve(dA, b, rtol=w.rtol, maxit=w.maxit, history=True)
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, g, rtol=w.rtol, maxit=w.maxit)
    lib = oracle.load_parallel()
    ref = oracle.cg(w.A.row_ptr, w.A.col_idx, w.A.values, w.b, rtol=w.rtol, maxit=w.maxit, history=True, lib=lib)
    assert info.status == ref["status"] == 0
    assert abs(info.iters - ref["iters"]) <= ITER_SLACK_F64
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"], k=50)
    adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, w.A.values, ref["x"], w.g, rtol=w.rtol, maxit=w.maxit, lib=lib)
    assert ainfo.status == adj["status"] == 0
    assert abs(ainfo.iters - adj["iters"]) <= ITER_SLACK_F64
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64


def _gpu_forward_adjoint(w, rtol, precond):
    """Forward solve with history and adjoint on the GPU; results copied to the host, device freed."""
    dA = to_dev(w.A)
    x, info, hist = sla.sla_cg_solve(dA, t(w.b), rtol=rtol, maxit=w.maxit, precond=precond, history=True)
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, t(w.g), rtol=rtol, maxit=w.maxit, precond=precond)
    out = (x.cpu().numpy(), hist.cpu().numpy(), gb.cpu().numpy(), gv.cpu().numpy(), info, ainfo)
    del dA, x, hist, gb, gv
    torch.cuda.empty_cache()
    return out


def _oracle_forward_adjoint(w, rtol, precond):
    lib = oracle.load_parallel()
    t0 = time.time()
    ref = oracle.cg(w.A.row_ptr, w.A.col_idx, w.A.values, w.b, rtol=rtol, maxit=w.maxit, precond=precond,
                    history=True, lib=lib)
    t1 = time.time()
    adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, w.A.values, ref["x"], w.g, rtol=rtol, maxit=w.maxit,
                            precond=precond, lib=lib)
    t2 = time.time()
    print(f"\n{w.name}: oracle on {lib.orc_threads(0)} host threads: forward {ref['iters']} iterations "
          f"{t1 - t0:.1f} s, adjoint {adj['iters']} iterations {t2 - t1:.1f} s")
    return ref, adj


def test_config4_jacobi_full_oracle():
    w = config4()
    xs, hs, gbs, gvs, info, ainfo = _gpu_forward_adjoint(w, w.rtol, 1)
    assert info.status == 0 and ainfo.status == 0, (info, ainfo)
    ref, adj = _oracle_forward_adjoint(w, w.rtol, 1)
    assert ref["status"] == adj["status"] == 0
    assert abs(info.iters - ref["iters"]) <= ITER_SLACK_F64
    assert abs(ainfo.iters - adj["iters"]) <= ITER_SLACK_F64
    assert rel(xs, ref["x"]) <= X_TOL_F64
    check_history(hs, ref["history"], k=50)
    assert gvs.shape == (w.A.nnz,)  # one gradient per stored entry, in CSR order: the pattern of A
    assert rel(gbs, adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gvs, adj["grad_values"]) <= GRAD_TOL_F64


@pytest.mark.skipif(_free_host_gb() < 64, reason="needs ~64 GB of host memory for the 169M-DOF oracle")
def test_config5_fixed_iterations_full_oracle():
    w = config5()
    assert w.A.row_ptr.dtype == np.int64
    xs, hs, gbs, gvs, info, ainfo = _gpu_forward_adjoint(w, 0.0, 0)
    assert info.status == sla.SLA_NOT_CONVERGED and info.iters == w.maxit
    assert ainfo.iters == w.maxit
    ref, adj = _oracle_forward_adjoint(w, 0.0, 0)
    assert ref["iters"] == adj["iters"] == w.maxit
    assert rel(xs, ref["x"]) <= X_TOL_F64
    check_history(hs, ref["history"], k=50)
    assert gvs.shape == (w.A.nnz,)
    assert rel(gbs, adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gvs, adj["grad_values"]) <= GRAD_TOL_F64


@pytest.mark.skipif(_free_host_gb() < 64, reason="needs ~40 GB of host memory for a 2.18e9-entry pattern")
def test_rowptr64_past_2_pow_31_entries():
    # 64-bit row offsets where they matter: 2,097,152 rows of up to 1,041 entries, 2.18e9 stored
    # entries (past 2^31), int64 row_ptr, through the engine AUTO picks (the graph loop at this
    # size).  Five CG iterations forward and adjoint (both stop at maxit), against the oracle's;
    # grad_values on sampled rows, among them the rows whose entries straddle and follow 2^31.
    from workloads import banded_dominant
    A = banded_dominant(1 << 21, 520)
    assert A.nnz > 2 ** 31 and A.row_ptr.dtype == np.int64
    rng = np.random.default_rng(71)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    rtol, maxit = 1e-12, 5
    dA = sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, A.values, "cuda:0")
    x, info, hist = sla.sla_cg_solve(dA, t(b), rtol=rtol, maxit=maxit, history=True)
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, t(g), rtol=rtol, maxit=maxit)
    lib = oracle.load_parallel()
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit, history=True, lib=lib)
    assert info.status == ref["status"] == 1 and info.iters == ref["iters"] == maxit
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"], k=maxit)
    # the adjoint of the symmetric solve: A lambda = g by the same CG from zero
    lam = oracle.cg(A.row_ptr, A.col_idx, A.values, g, rtol=rtol, maxit=maxit, lib=lib)["x"]
    assert ainfo.status == 1 and ainfo.iters == maxit
    assert rel(gb.cpu().numpy(), lam) <= GRAD_TOL_F64
    # grad_values[e] = -lambda_row(e) * x_col(e) on sampled rows
    r31 = int(np.searchsorted(A.row_ptr, 2 ** 31, side="right")) - 1  # the row holding entry 2^31
    rows = np.unique(np.concatenate([rng.choice(A.n, 300, replace=False), np.arange(r31 - 2, r31 + 3),
                                     np.arange(A.n - 3, A.n), [0, 1]]))
    ents = np.concatenate([np.arange(A.row_ptr[i], A.row_ptr[i + 1]) for i in rows])
    assert ents.max() > 2 ** 31
    want = np.concatenate([-lam[i] * ref["x"][A.col_idx[A.row_ptr[i]:A.row_ptr[i + 1]]] for i in rows])
    got = gv[torch.from_numpy(ents).to(gv.device)].cpu().numpy()
    assert rel(got, want) <= GRAD_TOL_F64
