"""The autograd node (CGSolve): gradients, finite differences, O(1) graph and memory independent of k."""
import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, to_dev, t, GRAD_TOL_F64
from workloads import diffusion_dirichlet, poisson_5pt

pytestmark = pytest.mark.gpu


def _problem(m=24, seed=3):
    A = diffusion_dirichlet(m, np.random.default_rng(seed).lognormal(0, 0.7, 2 * m * (m + 1)))
    rng = np.random.default_rng(seed + 1)
    return A, rng.standard_normal(A.n), rng.standard_normal(A.n)


@pytest.mark.parametrize("precond", [0, 1])
def test_solve_backward_matches_oracle_adjoint(precond):
    A, b, g = _problem()
    dA = to_dev(A)
    vals = dA.values.clone().requires_grad_(True)
    bt = t(b).requires_grad_(True)
    x = sla.solve(dA.with_values(vals), bt, rtol=1e-12, maxit=10000, precond=precond)
    (x * t(g)).sum().backward()
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-12, maxit=10000, precond=precond)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-12, maxit=10000, precond=precond)
    assert rel(bt.grad.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(vals.grad.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64


def test_symmetric_pair_finite_difference():
    # perturbing A_ij and A_ji together keeps A symmetric, so the forward CG stays valid:
    # dL/dh = gv_ij + gv_ji
    A, b, g = _problem(m=12, seed=9)
    dA = to_dev(A)
    vals = dA.values.clone().requires_grad_(True)
    x = sla.solve(dA.with_values(vals), t(b), rtol=1e-14, maxit=10000)
    (x * t(g)).sum().backward()
    gv = vals.grad.cpu().numpy()
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    for k in [3, 40, 200]:
        i, j = rows[k], A.col_idx[k]
        kk = [q for q in range(A.row_ptr[j], A.row_ptr[j + 1]) if A.col_idx[q] == i][0]
        h = 1e-5

        def L(delta):
            v = A.values.copy()
            v[k] += delta
            if kk != k:
                v[kk] += delta
            xx, info, _ = sla.sla_cg_solve(dA.with_values(t(v)), t(b), rtol=1e-14, maxit=10000)
            return float(xx.cpu().numpy() @ g)

        fd = (L(h) - L(-h)) / (2 * h)
        an = gv[k] + (gv[kk] if kk != k else 0.0)
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (k, fd, an)


def test_graph_is_one_node_and_memory_independent_of_iterations():
    A = poisson_5pt(200)
    dA = to_dev(A)
    b = t(np.random.default_rng(1).standard_normal(A.n))
    peaks = []
    for k in (20, 400):
        vals = dA.values.clone().requires_grad_(True)
        bt = b.clone().requires_grad_(True)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        with pytest.warns(UserWarning):
            x = sla.solve(dA.with_values(vals), bt, rtol=0.0, maxit=k)
        assert x.grad_fn is not None and type(x.grad_fn).__name__ == "CGSolveBackward"
        assert all(f[0] is None or type(f[0]).__name__ == "AccumulateGrad" for f in x.grad_fn.next_functions)
        with pytest.warns(UserWarning):
            x.sum().backward()
        torch.cuda.synchronize()
        peaks.append(torch.cuda.max_memory_allocated() - base)
        del x, vals, bt
    assert peaks[0] == peaks[1], peaks
    # O(n + nnz): well under 16 vectors of n doubles plus two value arrays
    assert peaks[1] <= 16 * A.n * 8 + 2 * A.nnz * 8 + (1 << 20)
