"""Gradient through the solve to physical coefficients on the GPU (autograd end to end).

Edge conductivities k = exp(theta) are assembled into the CSR values on the device with torch
ops (values = M k); x = solve(A, b) runs the CUDA CG and its backward the CUDA adjoint; the loss
L = 1/2 ||x - x_t||^2.  dL/dtheta must match the fp64 oracle's chain (adjoint solve,
grad_values = -lambda_i x_j, then M^T and the exp), and a few Adam steps must reduce L.
"""
import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, GRAD_TOL_F64
from inverse_helpers import edge_map, apply_map, apply_map_t

pytestmark = pytest.mark.gpu


def _setup(m, seed):
    E = 2 * m * (m + 1)
    base, rows, cols, wts = edge_map(m)
    rng = np.random.default_rng(seed)
    theta = rng.normal(0.0, 0.5, E)
    k_true = rng.lognormal(0.0, 0.5, E)
    b = rng.standard_normal(base.n)
    x_t = oracle.cg(base.row_ptr, base.col_idx, apply_map(base.nnz, rows, cols, wts, k_true), b, rtol=1e-14,
                    maxit=20000)["x"]
    dev = torch.device("cuda")
    Mi = torch.tensor(np.stack([rows, cols]), dtype=torch.int64, device=dev)
    M = torch.sparse_coo_tensor(Mi, torch.tensor(wts, device=dev), (base.nnz, E)).coalesce()
    return base, rows, cols, wts, theta, b, x_t, M, dev


def _loss(base, M, theta_t, b_t, x_t_t, dev):
    k = torch.exp(theta_t)
    vals = torch.sparse.mm(M, k[:, None])[:, 0]
    A = sla.CSRMatrix(torch.tensor(base.row_ptr, device=dev), torch.tensor(base.col_idx, device=dev), vals)
    x = sla.solve(A, b_t, rtol=1e-13, maxit=20000)
    d = x - x_t_t
    return 0.5 * (d * d).sum()


def test_coefficient_gradient_matches_oracle_chain():
    m = 24
    base, rows, cols, wts, theta, b, x_t, M, dev = _setup(m, 5)
    th = torch.tensor(theta, device=dev, requires_grad=True)
    L = _loss(base, M, th, torch.tensor(b, device=dev), torch.tensor(x_t, device=dev), dev)
    L.backward()
    k = np.exp(theta)
    vals = apply_map(base.nnz, rows, cols, wts, k)
    x = oracle.cg(base.row_ptr, base.col_idx, vals, b, rtol=1e-14, maxit=20000)["x"]
    adj = oracle.cg_adjoint(base.row_ptr, base.col_idx, vals, x, x - x_t, rtol=1e-14, maxit=20000)
    grad_theta = apply_map_t(2 * m * (m + 1), rows, cols, wts, adj["grad_values"]) * k
    assert float(L.detach()) == pytest.approx(0.5 * float((x - x_t) @ (x - x_t)), rel=1e-9)
    assert rel(th.grad.cpu().numpy(), grad_theta) <= GRAD_TOL_F64


def test_adam_on_coefficients_reduces_the_loss():
    m = 24
    base, rows, cols, wts, theta, b, x_t, M, dev = _setup(m, 6)
    th = torch.tensor(theta, device=dev, requires_grad=True)
    b_t, x_t_t = torch.tensor(b, device=dev), torch.tensor(x_t, device=dev)
    opt = torch.optim.Adam([th], lr=0.05)
    losses = []
    for _ in range(25):
        opt.zero_grad()
        L = _loss(base, M, th, b_t, x_t_t, dev)
        L.backward()
        opt.step()
        losses.append(float(L.detach()))
    assert all(np.isfinite(losses))
    assert losses[-1] < 0.5 * losses[0]
