"""The adjoint gradient carried to physical coefficients, on the CPU with the oracle.

Loss L(k) = 1/2 ||x(k) - x_t||^2 with A(k) x = b and A's values linear in the edge
conductivities k (values = M k).  The chain rule through the pattern gradient gives
dL/dk = M^T grad_values with grad_values = -lambda_i x_j from the adjoint solve A lambda = x - x_t
(the linear-system adjoint of the method: grad_A on the sparsity pattern).  Checked against
central finite differences of L computed by forward solves alone.
"""
import numpy as np
import pytest

import oracle
from inverse_helpers import edge_map, apply_map, apply_map_t


def test_coefficient_gradient_matches_finite_differences():
    m = 8
    E = 2 * m * (m + 1)
    base, rows, cols, wts = edge_map(m)
    rng = np.random.default_rng(11)
    k = rng.lognormal(0.0, 0.5, E)
    k_true = rng.lognormal(0.0, 0.5, E)
    b = rng.standard_normal(base.n)
    rp, ci = base.row_ptr, base.col_idx

    def solve(kk):
        return oracle.cg(rp, ci, apply_map(base.nnz, rows, cols, wts, kk), b, rtol=1e-14, maxit=10000)["x"]

    x_t = solve(k_true)

    def loss(kk):
        d = solve(kk) - x_t
        return 0.5 * float(d @ d)

    x = solve(k)
    adj = oracle.cg_adjoint(rp, ci, apply_map(base.nnz, rows, cols, wts, k), x, x - x_t, rtol=1e-14, maxit=10000)
    grad_k = apply_map_t(E, rows, cols, wts, adj["grad_values"])
    for j in (0, E // 3, E - 1, int(np.argmax(np.abs(grad_k)))):
        h = 1e-6 * k[j]
        kp, km = k.copy(), k.copy()
        kp[j] += h
        km[j] -= h
        fd = (loss(kp) - loss(km)) / (2 * h)
        assert fd == pytest.approx(grad_k[j], rel=1e-5, abs=1e-12 * max(1.0, np.abs(grad_k).max()))


def test_edge_map_reproduces_the_generator():
    from workloads import diffusion_dirichlet
    m = 6
    E = 2 * m * (m + 1)
    base, rows, cols, wts = edge_map(m)
    k = np.random.default_rng(3).lognormal(0.0, 1.0, E)
    # equal up to the order in which an entry's edge contributions are added
    assert np.allclose(apply_map(base.nnz, rows, cols, wts, k), diffusion_dirichlet(m, k).values, rtol=4e-16, atol=0)
