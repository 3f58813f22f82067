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


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_solve_batched_backward(dtype):
    # the batched autograd node: forward and backward are the batched solve and adjoint, bit for bit,
    # and each system matches the oracle (its adjoint chained from the oracle's own x)
    from workloads import config3
    from gpu_helpers import TOL_F32, X_TOL_F64
    w = config3(m=24, batch=5)
    rtol = 1e-10 if dtype == np.float64 else w.rtol
    rp = torch.from_numpy(w.A.row_ptr).cuda()
    ci = torch.from_numpy(w.A.col_idx).cuda()
    vals = torch.from_numpy(w.values_b.astype(dtype)).cuda().requires_grad_(True)
    b = torch.from_numpy(w.b.astype(dtype)).cuda().requires_grad_(True)
    g = torch.from_numpy(w.g.astype(dtype)).cuda()
    x = sla.solve_batched(rp, ci, vals, b, rtol=rtol, maxit=5000)
    x.backward(g)
    P = sla.CSRMatrix(rp, ci, vals.detach()[0])
    xd, _, _ = sla.sla_cg_solve_batched(P, vals.detach(), b.detach(), rtol=rtol, maxit=5000)
    gbd, gvd, _ = sla.sla_cg_adjoint_batched(P, vals.detach(), xd, g, rtol=rtol, maxit=5000)
    assert torch.equal(x.detach(), xd) and torch.equal(b.grad, gbd) and torch.equal(vals.grad, gvd)
    tol_x = X_TOL_F64 if dtype == np.float64 else TOL_F32
    tol_g = GRAD_TOL_F64 if dtype == np.float64 else TOL_F32
    for s in range(w.batch):
        v64 = w.values_b[s].astype(dtype).astype(np.float64)
        b64, g64 = w.b[s].astype(dtype).astype(np.float64), w.g[s].astype(dtype).astype(np.float64)
        ref = oracle.cg(w.A.row_ptr, w.A.col_idx, v64, b64, rtol=rtol, maxit=5000)
        adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, v64, ref["x"], g64, rtol=rtol, maxit=5000)
        assert rel(x[s].detach().cpu().numpy(), ref["x"]) <= tol_x
        assert rel(b.grad[s].cpu().numpy(), adj["grad_b"]) <= tol_g
        assert rel(vals.grad[s].cpu().numpy(), adj["grad_values"]) <= tol_g


def test_method_style_interface():
    # A.solve(b), A.matvec(x), A.eigsh(): the module functions, with their gradients
    A, b, g = _problem(m=16, seed=5)
    dA = to_dev(A)
    v1 = dA.values.clone().requires_grad_(True)
    v2 = dA.values.clone().requires_grad_(True)
    x1 = dA.with_values(v1).solve(t(b), rtol=1e-12)
    x2 = sla.solve(dA.with_values(v2), t(b), rtol=1e-12)
    (x1 * t(g)).sum().backward()
    (x2 * t(g)).sum().backward()
    assert torch.equal(x1.detach(), x2.detach()) and torch.equal(v1.grad, v2.grad)
    assert torch.equal(dA.matvec(t(b)), sla.matvec(dA, t(b)))
    mu1, _ = dA.eigsh()
    mu2, _ = sla.eigsh_smallest(dA)
    assert float(mu1.detach()) == float(mu2.detach())
