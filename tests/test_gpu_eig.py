"""Eigenvalue problems on the GPU against the fp64 oracle.

The gradient kernel (d mu / d A_ij = v_i v_j on the pattern, weighted over k eigenvectors) is
compared with the oracle on arbitrary vectors entry by entry, within the rounding bound of the
sum: each side forms k products of three factors and k - 1 additions in fp64, so each is within
(k + 1) u sum_s |w_s v_s[i] v_s[j]| of the exact value (u = 2^-53) and the two within twice that;
for float data one float ulp of the result is added (each side rounds its fp64 value once).  The eigenpair from inverse iteration is compared
with the oracle's dense symmetric eigensolver and with the five-point Laplacian's closed form, to
tolerances derived from the stopping test: a unit vector with ||A v - mu v|| <= tol * mu is within
tol * mu / gap of the eigenvector (sin theta bound), and its Rayleigh quotient within
(tol * mu)^2 / gap of the eigenvalue, plus rounding.
"""
import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, to_dev, t
from oracle_pins import poisson_fundamental
from workloads import poisson_5pt, diffusion_dirichlet, random_spd

pytestmark = pytest.mark.gpu

EPS64 = np.finfo(np.float64).eps
EPS32 = float(np.finfo(np.float32).eps)


def assert_eig_grad_close(gv, rp, ci, V, w, dtype):
    """gv against the oracle's sum_s w_s (v_s[i] v_s[j]), entry by entry, within the rounding bound."""
    V64 = np.atleast_2d(np.asarray(V, dtype=np.float64))
    k = V64.shape[0]
    ref = oracle.eig_grad_values(rp, ci, V64, w)
    rows = np.repeat(np.arange(len(rp) - 1), np.diff(np.asarray(rp, dtype=np.int64)))
    wv = np.ones(k) if w is None else np.asarray(w, dtype=np.float64)
    terms = np.zeros(len(ci))
    for s in range(k):
        terms += np.abs(wv[s] * V64[s, rows] * V64[s, ci])
    bound = (k + 1) * EPS64 * terms + 1e-300
    if dtype == np.float32:
        bound = bound + EPS32 * np.abs(ref)
    diff = np.abs(np.asarray(gv, dtype=np.float64) - ref)
    assert np.all(diff <= bound), f"max excess {np.max(diff / bound):.3g} of the rounding bound"


def _vec_bound(tol, mu, gap, n, eps=EPS64):
    return 10.0 * tol * mu / gap + 100.0 * np.sqrt(n) * eps


# --------------------------------------------------------------------------- gradient kernel

@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("k", [1, 3, 16])
def test_eig_grad_values_within_rounding(dtype, k):
    A = random_spd(777, 5.0, 3, long_rows=2)
    rng = np.random.default_rng(40 + k)
    V = rng.standard_normal((k, A.n)).astype(dtype)
    w = rng.standard_normal(k)
    gv = sla.sla_eig_grad_values(to_dev(A, dtype), t(V), weights=w).cpu().numpy()
    assert gv.dtype == dtype
    assert_eig_grad_close(gv, A.row_ptr, A.col_idx, V, w, dtype)
    # unit weights by default; k = 0 gives zeros
    gv1 = sla.sla_eig_grad_values(to_dev(A, dtype), t(V[:1])).cpu().numpy()
    assert_eig_grad_close(gv1, A.row_ptr, A.col_idx, V[:1], None, dtype)
    z = sla.sla_eig_grad_values(to_dev(A, dtype), t(np.zeros((0, A.n), dtype))).cpu().numpy()
    assert not z.any()


def test_eig_grad_values_ragged_rows_int64():
    # rows of length 0..40 and an int64 row_ptr, several warps' worth of row groups with a ragged tail
    rng = np.random.default_rng(9)
    n = 32 * 37 + 5
    lens = rng.integers(0, 41, n)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ci = np.concatenate([np.sort(rng.choice(n, L, replace=False)) for L in lens]).astype(np.int32)
    vals = rng.standard_normal(rp[-1])
    dA = sla.CSRMatrix.from_numpy(rp, ci, vals, "cuda:0")
    V = rng.standard_normal((2, n))
    gv = sla.sla_eig_grad_values(dA, t(V), weights=[0.5, -2.0]).cpu().numpy()
    assert_eig_grad_close(gv, rp, ci, V, [0.5, -2.0], np.float64)


# --------------------------------------------------------------------------- eigenpair

@pytest.mark.parametrize("m", [16, 32])
def test_eig_smallest_poisson_closed_form(m):
    A = poisson_5pt(m)
    mu, v, info = sla.sla_eig_smallest(to_dev(A), tol=1e-10)
    mu0, v0 = poisson_fundamental(m)
    th = np.pi / (m + 1)
    gap = 2.0 * (np.cos(th) - np.cos(2 * th))
    assert info.status == sla.SLA_OK and info.iters > 0
    assert info.residual <= 1e-10 * info.mu
    assert abs(mu - mu0) <= 1e-12 * mu0 + 20 * EPS64 * 8.0
    assert np.linalg.norm(v.cpu().numpy() - v0) <= _vec_bound(1e-10, mu0, gap, A.n)


@pytest.mark.parametrize("precond", [0, 1])
@pytest.mark.parametrize("loop", [sla.SLA_LOOP_AUTO, sla.SLA_LOOP_GRAPH, sla.SLA_LOOP_RESIDENT])
def test_eig_smallest_matches_dense_oracle(loop, precond):
    m = 30
    A = diffusion_dirichlet(m, np.random.default_rng(17).lognormal(0.0, 0.5, 2 * m * (m + 1)))
    mu_o, V_o = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 2)
    gap = mu_o[1] - mu_o[0]
    tol = 1e-10
    mu, v, info = sla.sla_eig_smallest(to_dev(A), tol=tol, precond=precond, loop=loop)
    assert info.status == sla.SLA_OK, info
    assert abs(mu - mu_o[0]) <= 1e-11 * mu_o[0]
    vg = v.cpu().numpy()
    assert abs(np.linalg.norm(vg) - 1.0) <= 1e-13
    assert vg.sum() >= 0.0  # sign convention, as the oracle's
    assert np.linalg.norm(vg - V_o[0]) <= _vec_bound(tol, mu_o[0], gap, A.n)


def test_eig_smallest_int64_rowptr_and_ragged_grid():
    # int64 row pointers; a 45 x 45 grid (2025 rows: several blocks with a ragged tail)
    m = 45
    A = poisson_5pt(m, rowptr64=True)
    assert A.row_ptr.dtype == np.int64
    mu, v, info = sla.sla_eig_smallest(to_dev(A), tol=1e-10)
    mu0, v0 = poisson_fundamental(m)
    th = np.pi / (m + 1)
    gap = 2.0 * (np.cos(th) - np.cos(2 * th))
    assert info.status == sla.SLA_OK, info
    assert abs(mu - mu0) <= 1e-11 * mu0
    assert np.linalg.norm(v.cpu().numpy() - v0) <= _vec_bound(1e-10, mu0, gap, A.n)
    gv = sla.sla_eig_grad_values(to_dev(A), v, weights=[-1.5]).cpu().numpy()
    assert_eig_grad_close(gv, A.row_ptr, A.col_idx, v.cpu().numpy(), [-1.5], np.float64)


def test_eig_smallest_float32():
    m = 24
    A = poisson_5pt(m)
    mu, v, info = sla.sla_eig_smallest(to_dev(A, np.float32), tol=1e-5)
    mu0, v0 = poisson_fundamental(m)
    assert info.status == sla.SLA_OK, info
    assert abs(mu - mu0) <= 1e-4 * mu0
    assert rel(v.cpu().numpy(), v0) <= 1e-3


def test_eig_smallest_status_cases():
    A = poisson_5pt(10)
    dA = to_dev(A)
    # a zero start vector: no direction to iterate on
    _, _, info = sla.sla_eig_smallest(dA, v0=torch.zeros(A.n, dtype=torch.float64, device="cuda:0"))
    assert info.status == sla.SLA_BREAKDOWN and info.iters == 0
    # negative definite: the first Rayleigh quotient is negative, before any solve
    neg = sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, -A.values, "cuda:0")
    _, _, info = sla.sla_eig_smallest(neg)
    assert info.status == sla.SLA_BREAKDOWN and info.iters == 0 and info.inner_iters == 0
    # maxit = 0: the start vector, normalised, with its Rayleigh quotient and residual
    v0 = np.random.default_rng(2).standard_normal(A.n)
    mu, v, info = sla.sla_eig_smallest(dA, v0=t(v0), maxit=0)
    assert info.status == sla.SLA_NOT_CONVERGED and info.iters == 0
    u = v0 / np.linalg.norm(v0)
    u = u if u.sum() >= 0 else -u
    assert np.allclose(v.cpu().numpy(), u, rtol=0, atol=1e-15)
    Au = oracle.spmv(A.row_ptr, A.col_idx, A.values, u)
    assert abs(mu - u @ Au) <= 1e-13 * abs(u @ Au)
    assert abs(info.residual - np.linalg.norm(Au - (u @ Au) * u)) <= 1e-12 * np.linalg.norm(Au)
    # an invalid option is rejected before any launch
    with pytest.raises(sla.SlaError):
        sla.sla_eig_smallest(dA, inner_factor=1.5)


# --------------------------------------------------------------------------- autograd

def test_eigsh_smallest_gradient():
    m = 20
    A = diffusion_dirichlet(m, np.random.default_rng(5).lognormal(0.0, 0.5, 2 * m * (m + 1)))
    vals = t(A.values).requires_grad_(True)
    dA = sla.CSRMatrix(t(A.row_ptr), t(A.col_idx), vals)
    mu, v = sla.eigsh_smallest(dA, tol=1e-11)
    assert not v.requires_grad
    (3.0 * mu).backward()
    mu_o, V_o = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 2)
    assert abs(float(mu.detach()) - mu_o[0]) <= 1e-11 * mu_o[0]
    ref = 3.0 * oracle.eig_grad_values(A.row_ptr, A.col_idx, V_o[:1])
    assert rel(vals.grad.cpu().numpy(), ref) <= 1e-8


# --------------------------------------------------------------------------- full size

@pytest.mark.slow
def test_eig_smallest_poisson1000_sampled():
    # 1M unknowns: the eigenpair against the closed form, the eigenvector on a sample of entries
    m = 1000
    A = poisson_5pt(m)
    tol = 1e-10
    mu, v, info = sla.sla_eig_smallest(to_dev(A), tol=tol)
    th = np.pi / (m + 1)
    mu0 = 4.0 - 4.0 * np.cos(th)
    gap = 2.0 * (np.cos(th) - np.cos(2 * th))
    assert info.status == sla.SLA_OK, info
    assert abs(mu - mu0) <= 1e-9 * mu0
    idx = np.random.default_rng(3).choice(A.n, 2000, replace=False)
    a, b = idx // m, idx % m
    s = np.sin(th * np.arange(1, m + 1))
    v0 = s[a] * s[b] / float(np.sum(s * s))
    vg = v.cpu().numpy()[idx]
    assert np.max(np.abs(vg - v0)) <= _vec_bound(tol, mu0, gap, A.n)
    # its gradient through autograd equals v_i v_j on a sample of stored entries
    gv = sla.sla_eig_grad_values(to_dev(A), v).cpu().numpy()
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    vv = v.cpu().numpy()
    e = np.random.default_rng(4).choice(A.nnz, 2000, replace=False)
    # one eigenvector with unit weight: a single rounded product v_i * v_j on both sides, so exact
    assert np.array_equal(gv[e], vv[rows[e]] * vv[A.col_idx[e]])


# --------------------------------------------------------------------------- k smallest eigenpairs

def _diffusion(m, seed):
    return diffusion_dirichlet(m, np.random.default_rng(seed).lognormal(0.0, 0.5, 2 * m * (m + 1)))


@pytest.mark.parametrize("loop", [sla.SLA_LOOP_AUTO, sla.SLA_LOOP_GRAPH])
@pytest.mark.parametrize("precond", [0, 1])
@pytest.mark.parametrize("k", [1, 3, 6])
def test_eigsh_k_matches_dense_oracle(k, precond, loop):
    # distinct eigenvalues: each eigenvector is unique up to sign (both sides take sum_i v_i >= 0).
    # AUTO: the k inner solves one by one; GRAPH: together in the batched CG
    A = _diffusion(20, 17)
    mu_o, V_o = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, k + 1)
    tol = 1e-10
    mu, V, info = sla.sla_eigsh(to_dev(A), k, tol=tol, precond=precond, loop=loop)
    assert info.status == sla.SLA_OK, info
    assert info.residual <= tol * float(mu[-1])
    Vg = V.cpu().numpy()
    assert np.linalg.norm(Vg @ Vg.T - np.eye(k)) <= 1e-12
    for s in range(k):
        gap = min(mu_o[s + 1] - mu_o[s], mu_o[s] - mu_o[s - 1] if s > 0 else np.inf)
        assert abs(float(mu[s]) - mu_o[s]) <= 1e-11 * mu_o[s]
        assert Vg[s].sum() >= 0.0
        assert np.linalg.norm(Vg[s] - V_o[s]) <= _vec_bound(tol, mu_o[s], gap, A.n)


def test_eigsh_poisson_multiple_eigenvalue():
    # the five-point Laplacian's 2nd and 3rd eigenvalues are equal (modes (1,2) and (2,1)): the
    # eigenvalues are unique, the vectors only up to a basis of that eigenspace
    m = 16
    A = poisson_5pt(m)
    th = np.pi / (m + 1)
    lam = lambda p, q: 4.0 - 2.0 * np.cos(p * th) - 2.0 * np.cos(q * th)  # noqa: E731
    exact = np.array([lam(1, 1), lam(1, 2), lam(2, 1), lam(2, 2)])
    mu, V, info = sla.sla_eigsh(to_dev(A), 4, tol=1e-10)
    assert info.status == sla.SLA_OK, info
    assert np.all(np.abs(mu.numpy() - exact) <= 1e-11 * exact)
    mu_o, V_o = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 5)
    Vg = V.cpu().numpy()
    P, P_o = Vg[1:3].T @ Vg[1:3], V_o[1:3].T @ V_o[1:3]  # projectors onto the double eigenspace
    gap = min(exact[1] - exact[0], exact[3] - exact[1])
    assert np.linalg.norm(P - P_o) <= 2 * _vec_bound(1e-10, exact[1], gap, A.n)
    for s in (0, 3):
        assert np.linalg.norm(Vg[s] - V_o[s]) <= _vec_bound(1e-10, exact[s], gap, A.n)


def test_eigsh_gradient_of_weighted_eigenvalues():
    A = _diffusion(16, 23)
    k, w = 3, np.array([1.5, -0.5, 2.0])
    vals = t(A.values).requires_grad_(True)
    dA = sla.CSRMatrix(t(A.row_ptr), t(A.col_idx), vals)
    mu, V = sla.eigsh(dA, k, tol=1e-11)
    assert mu.requires_grad and not V.requires_grad
    (mu * t(w)).sum().backward()
    mu_o, V_o = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, k + 1)
    assert np.all(np.abs(mu.detach().cpu().numpy() - mu_o[:k]) <= 1e-11 * mu_o[:k])
    ref = oracle.eig_grad_values(A.row_ptr, A.col_idx, V_o[:k], w)
    assert rel(vals.grad.cpu().numpy(), ref) <= 1e-8
    # the same through the method-style interface
    mu2, _ = dA.eigsh(k=k, tol=1e-11)
    assert torch.allclose(mu2.detach(), mu.detach(), rtol=1e-12, atol=0)


def test_eigsh_k1_agrees_with_eig_smallest():
    A = _diffusion(24, 7)
    mu1, v1, _ = sla.sla_eig_smallest(to_dev(A), tol=1e-11)
    mu, V, info = sla.sla_eigsh(to_dev(A), 1, tol=1e-11)
    assert info.status == sla.SLA_OK
    assert abs(float(mu[0]) - mu1) <= 1e-12 * mu1
    assert np.linalg.norm(V[0].cpu().numpy() - v1.cpu().numpy()) <= 1e-8


def test_eigsh_float32():
    m = 20
    A = poisson_5pt(m)
    th = np.pi / (m + 1)
    mu, V, info = sla.sla_eigsh(to_dev(A, np.float32), 2, tol=1e-5)
    assert info.status == sla.SLA_OK, info
    exact = np.array([4.0 - 4.0 * np.cos(th), 4.0 - 2.0 * np.cos(th) - 2.0 * np.cos(2 * th)])
    assert np.all(np.abs(mu.numpy() - exact) <= 1e-4 * exact)
    assert V.dtype == torch.float32


def test_eigsh_status_and_argument_cases():
    A = poisson_5pt(10)
    dA = to_dev(A)
    for k in (0, 17, A.n + 1):
        with pytest.raises(sla.SlaError):
            sla.sla_eigsh(dA, k, V0=None if k == 0 or k > 16 else torch.zeros(k, A.n, dtype=torch.float64,
                                                                              device="cuda:0"))
    # a rank-deficient start block: two equal rows
    V0 = np.random.default_rng(1).standard_normal((3, A.n))
    V0[2] = V0[1]
    _, _, info = sla.sla_eigsh(dA, 3, V0=t(V0))
    assert info.status == sla.SLA_BREAKDOWN and info.iters == 0
    # negative definite: the first Ritz values are negative, before any solve
    neg = sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, -A.values, "cuda:0")
    _, _, info = sla.sla_eigsh(neg, 2)
    assert info.status == sla.SLA_BREAKDOWN and info.iters == 0 and info.inner_iters == 0
    # maxit = 0: the Ritz pairs of the start block, not converged
    mu, V, info = sla.sla_eigsh(dA, 2, maxit=0)
    assert info.status == sla.SLA_NOT_CONVERGED and info.iters == 0
    Vg = V.cpu().numpy()
    assert np.linalg.norm(Vg @ Vg.T - np.eye(2)) <= 1e-12
