"""Pins of the fp64 oracle against facts fixed by the mathematics, not by the oracle itself.

Each pin is a function ``pin_xxx(lib)`` that raises AssertionError when the
oracle library ``lib`` (see ``oracle.load``) disagrees with:

  * dense linear algebra on tiny grids (numpy.linalg.solve / exact rational
    elimination with ``fractions.Fraction``);
  * the closed-form eigenvalues of the five-point Laplacian,
    4 - 2cos(i pi/(m+1)) - 2cos(j pi/(m+1)), and the CG iteration bound that
    follows from the condition number;
  * finite termination of CG after (number of distinct eigenvalues) steps;
  * the relation between the recursively updated residual and the true
    residual b - A x_k of the returned iterate;
  * the adjoint identity <g, A^{-1} c> = <A^{-T} g, c>;
  * central finite differences of L = <g, x(A, b)> with respect to b and to a
    single stored entry of A (re-solved densely, since the perturbed matrix is
    not symmetric);
  * the exact scaling invariants sum_k gv_k values_k = -<g, x> and
    <grad_b, b> = <g, x> (from x(tA) = x/t and x(tb) = t x);
  * for eigenvalue problems: the closed-form fundamental mode of the
    five-point Laplacian, central differences of eigenvalues of the perturbed
    (non-symmetric) matrix, and the identity sum_e gv_e A_e = v^T A v = mu;
  * the Jacobi special case: with constant diagonal 4 the preconditioned
    iterates equal the unpreconditioned ones bit for bit (scaling by 1/4 is
    exact in binary floating point), and in general Jacobi PCG iterates equal
    D^{-1/2} times the plain CG iterates of the symmetrically scaled system.

The method is that of "torch-sla" (Chi, Wen), technical summary, Methodology
section 2 (adjoint differentiation framework, linear systems and eigenvalue
problems).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle
from workloads import poisson_5pt, diffusion_dirichlet, diffusion_interior, random_spd, config1, convection_diffusion

EPS = np.finfo(np.float64).eps


def poisson_eigs(m: int) -> np.ndarray:
    th = np.arange(1, m + 1) * np.pi / (m + 1)
    return (4.0 - 2.0 * np.cos(th)[:, None] - 2.0 * np.cos(th)[None, :]).reshape(-1)


def poisson_kappa(m: int) -> float:
    th = np.pi / (m + 1)
    lmin = 4.0 - 4.0 * np.cos(th)
    lmax = 4.0 + 4.0 * np.cos(th)
    return lmax / lmin


def cg_residual_bound(kappa: float, rtol: float) -> int:
    """Smallest k with 2 sqrt(kappa) ((sqrt(kappa)-1)/(sqrt(kappa)+1))^k <= rtol (x0 = 0)."""
    s = math.sqrt(kappa)
    return int(math.ceil(math.log(2.0 * s / rtol) / math.log((s + 1.0) / (s - 1.0))))


# --------------------------------------------------------------------------- spmv / dot

def pin_spmv_dense(lib):
    for n, seed, hubs in [(1, 0, 0), (2, 1, 0), (17, 2, 0), (33, 3, 2), (257, 4, 3)]:
        A = random_spd(n, 4.0, seed, long_rows=hubs)
        x = np.random.default_rng(seed + 100).standard_normal(n)
        y = oracle.spmv(A.row_ptr, A.col_idx, A.values, x, lib=lib)
        D = A.dense()
        yd = D @ x
        bound = 4 * np.diff(A.row_ptr.astype(np.int64)).max() * EPS * (np.abs(D) @ np.abs(x)) + 1e-300
        assert np.all(np.abs(y - yd) <= bound), (n, np.max(np.abs(y - yd) / bound))


def pin_spmv_exact_integers(lib):
    # small integers: every product and partial sum is exact, so y must equal the dense product exactly
    A = poisson_5pt(7)
    x = np.random.default_rng(5).integers(-50, 50, A.n).astype(np.float64)
    y = oracle.spmv(A.row_ptr, A.col_idx, A.values, x, lib=lib)
    assert np.array_equal(y, A.dense() @ x)
    # empty matrix
    y0 = oracle.spmv(np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0), np.zeros(0), lib=lib)
    assert y0.shape == (0,)


def pin_dot(lib):
    rng = np.random.default_rng(7)
    # lengths around and across the multi-core build's 4096-entry chunks
    for n in [0, 1, 5, 1000, 4095, 4096, 4097, 3 * 4096 + 17, 20000]:
        a, b = rng.standard_normal(n), rng.standard_normal(n)
        exact = math.fsum((a * b).tolist()) if n else 0.0
        got = oracle.dot(a, b, lib=lib)
        assert abs(got - exact) <= n * EPS * float(np.abs(a) @ np.abs(b)) + 1e-300
    assert oracle.dot(np.array([3.0, 4.0]), np.array([5.0, -2.0]), lib=lib) == 7.0
    # small integers: every partial sum is exact whatever the order, so the result is exact
    for n in [4097, 2 * 4096, 10000]:
        a = rng.integers(-20, 21, n).astype(np.float64)
        b = rng.integers(-20, 21, n).astype(np.float64)
        assert oracle.dot(a, b, lib=lib) == float(int(a.astype(np.int64) @ b.astype(np.int64)))


def pin_cg_several_chunks_true_residual(lib):
    # a system longer than two dot-product chunks (n = 4900): the returned iterate's true residual,
    # computed with scipy's sparse product (not the oracle's), meets the stopping rule up to the
    # usual drift of the recursive residual, and the solution agrees with a sparse direct solve
    sp = __import__("pytest").importorskip("scipy.sparse")
    spla = __import__("pytest").importorskip("scipy.sparse.linalg")
    m = 70
    A = diffusion_dirichlet(m, np.random.default_rng(61).lognormal(0, 0.5, 2 * m * (m + 1)))
    S = sp.csr_matrix((A.values, A.col_idx, A.row_ptr.astype(np.int64)), shape=(A.n, A.n))
    b = np.random.default_rng(62).standard_normal(A.n)
    for precond in (0, 1):
        r = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=5000, precond=precond, lib=lib)
        assert r["status"] == 0
        true_rel = np.linalg.norm(b - S @ r["x"]) / np.linalg.norm(b)
        assert true_rel <= 1.5e-10, (precond, true_rel)
        xd = spla.spsolve(S.tocsc(), b)
        assert np.linalg.norm(r["x"] - xd) <= 1e-10 * 1e4 * np.linalg.norm(xd)


def _random_csr(n, per_row, seed):
    """A structurally non-symmetric random CSR matrix (sorted, unique columns per row)."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i in range(n):
        k = int(rng.integers(0, per_row + 1)) if n else 0
        c = np.sort(rng.choice(n, min(k, n), replace=False))
        rows.append(np.full(c.shape[0], i))
        cols.append(c)
    cols = np.concatenate(cols).astype(np.int32) if n else np.zeros(0, np.int32)
    lens = np.array([c.shape[0] for c in rows]) if n else np.zeros(0, np.int64)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    vals = rng.standard_normal(cols.shape[0])
    return rp, cols, vals


def _dense(rp, ci, v, n):
    D = np.zeros((n, n))
    for i in range(n):
        for e in range(rp[i], rp[i + 1]):
            D[i, ci[e]] += v[e]
    return D


def pin_spmv_transpose_dense(lib):
    for n, per_row, seed in [(1, 1, 0), (7, 3, 1), (40, 6, 2), (300, 9, 3)]:
        rp, ci, v = _random_csr(n, per_row, seed)
        D = _dense(rp, ci, v, n)
        assert not np.array_equal(D, D.T) or n == 1  # a genuinely non-symmetric case
        x = np.random.default_rng(seed + 50).standard_normal(n)
        y = oracle.spmv_transpose(rp, ci, v, x, lib=lib)
        bound = 4 * max(per_row, 1) * EPS * (np.abs(D.T) @ np.abs(x)) + 1e-300
        assert np.all(np.abs(y - D.T @ x) <= bound * n), n
    # small integers: exact
    rp, ci, v = _random_csr(60, 5, 9)
    v = np.round(v * 10)
    x = np.random.default_rng(8).integers(-9, 10, 60).astype(np.float64)
    assert np.array_equal(oracle.spmv_transpose(rp, ci, v, x, lib=lib), _dense(rp, ci, v, 60).T @ x)
    # the adjoint identity <g, A x> = <A^T g, x>
    rp, ci, v = _random_csr(200, 7, 4)
    g, x = np.random.default_rng(5).standard_normal(200), np.random.default_rng(6).standard_normal(200)
    lhs = float(g @ oracle.spmv(rp, ci, v, x, lib=lib))
    rhs = float(oracle.spmv_transpose(rp, ci, v, g, lib=lib) @ x)
    assert abs(lhs - rhs) <= 1e-12 * (np.abs(g) @ np.abs(_dense(rp, ci, v, 200)) @ np.abs(x))


def pin_matvec_grad_values(lib):
    # L = <g, A x> is linear in each stored value: dL/dv_k = g_row x_col exactly, and
    # sum_k gv_k v_k = <g, A x>; a central difference reproduces an entry to rounding
    n = 50
    rp, ci, v = _random_csr(n, 6, 11)
    rng = np.random.default_rng(12)
    g, x = rng.standard_normal(n), rng.standard_normal(n)
    gv = oracle.matvec_grad_values(rp, ci, g, x, lib=lib)
    rows = np.repeat(np.arange(n), np.diff(rp))
    assert np.array_equal(gv, g[rows] * x[ci])
    L = float(g @ (_dense(rp, ci, v, n) @ x))
    assert abs(float(gv @ v) - L) <= 1e-12 * (np.abs(g) @ np.abs(_dense(rp, ci, v, n)) @ np.abs(x))
    for k in (0, int(ci.shape[0]) // 2, int(ci.shape[0]) - 1):
        h = 1e-3
        vp, vm = v.copy(), v.copy()
        vp[k] += h
        vm[k] -= h
        fd = (float(g @ (_dense(rp, ci, vp, n) @ x)) - float(g @ (_dense(rp, ci, vm, n) @ x))) / (2 * h)
        assert abs(fd - gv[k]) <= 1e-9 * max(1.0, abs(gv[k]))


# --------------------------------------------------------------------------- forward CG

def pin_cg_vs_dense(lib):
    cases = []
    for m in [2, 3, 4, 8, 16, 24]:
        cases.append(("poisson", poisson_5pt(m)))
    rng = np.random.default_rng(11)
    cases.append(("interior", diffusion_interior(9, rng.lognormal(0, 0.5, 2 * 9 * 8), 0.01)))
    cases.append(("dirichlet", diffusion_dirichlet(10, rng.lognormal(0, 1.0, 2 * 10 * 11))))
    cases.append(("random", random_spd(150, 5.0, 3, long_rows=2)))
    for name, A in cases:
        b = np.random.default_rng(A.n).standard_normal(A.n)
        D = A.dense()
        xs = np.linalg.solve(D, b)
        ev = np.linalg.eigvalsh(D)
        kappa = ev[-1] / ev[0]
        for precond in (0, 1):
            out = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-12, maxit=10000, precond=precond, lib=lib)
            assert out["status"] == 0, (name, precond, out["status"])
            err = np.linalg.norm(out["x"] - xs) / np.linalg.norm(xs)
            assert err <= kappa * 1e-12 * 4 + 1e-13, (name, precond, err)
            true_res = np.linalg.norm(b - D @ out["x"]) / np.linalg.norm(b)
            assert true_res <= 1e-11, (name, precond, true_res)


def pin_cg_exact_rational(lib):
    # m = 2 Poisson: A^{-1} e1 = (7/24, 1/12, 1/12, 1/24), solved exactly over the rationals here
    A = poisson_5pt(2)
    D = [[Fraction(int(v)) for v in row] for row in A.dense()]
    b = [Fraction(1), Fraction(0), Fraction(0), Fraction(0)]
    n = 4
    M = [row[:] + [b[i]] for i, row in enumerate(D)]
    for c in range(n):
        piv = next(r for r in range(c, n) if M[r][c] != 0)
        M[c], M[piv] = M[piv], M[c]
        for r in range(n):
            if r != c and M[r][c] != 0:
                f = M[r][c] / M[c][c]
                M[r] = [M[r][k] - f * M[c][k] for k in range(n + 1)]
    x_exact = [M[i][n] / M[i][i] for i in range(n)]
    assert x_exact == [Fraction(7, 24), Fraction(1, 12), Fraction(1, 12), Fraction(1, 24)]
    out = oracle.cg(A.row_ptr, A.col_idx, A.values, np.array([1.0, 0, 0, 0]), rtol=0.0, maxit=3, lib=lib)
    assert np.max(np.abs(out["x"] - np.array([float(v) for v in x_exact]))) <= 8 * EPS
    # m = 1: A = [4], one step gives b/4 exactly
    A1 = poisson_5pt(1)
    out1 = oracle.cg(A1.row_ptr, A1.col_idx, A1.values, np.array([3.0]), rtol=1e-14, maxit=10, lib=lib)
    assert out1["iters"] == 1 and out1["x"][0] == 0.75 and out1["status"] == 0


def pin_finite_termination(lib):
    # CG terminates in at most (number of distinct eigenvalues) steps in exact arithmetic
    for m in [2, 3, 4, 5]:
        A = poisson_5pt(m)
        ev = poisson_eigs(m)
        distinct = len(np.unique(np.round(ev, 9)))
        b = np.random.default_rng(m).standard_normal(A.n)
        out = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=distinct, history=True, lib=lib)
        assert out["rel_res"] < 1e-12, (m, distinct, out["rel_res"])
        # and not before: with all eigen-components present one step fewer leaves a visible residual
        out2 = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=distinct - 1, lib=lib)
        assert out2["rel_res"] > 1e-10, (m, out2["rel_res"])


def pin_eigen_closed_form_and_bound(lib):
    for m in [3, 8, 16]:
        A = poisson_5pt(m)
        ev = np.linalg.eigvalsh(A.dense())
        assert np.max(np.abs(np.sort(poisson_eigs(m)) - ev)) <= 1e-12
    # iteration count within the residual bound derived from kappa (config 1: m = 64, rtol 1e-10)
    w = config1()
    out = oracle.cg(w.A.row_ptr, w.A.col_idx, w.A.values, w.b, rtol=w.rtol, maxit=w.maxit, lib=lib)
    kappa = poisson_kappa(64)
    assert abs(kappa - 1711.7) < 0.1
    assert out["status"] == 0 and 0 < out["iters"] <= cg_residual_bound(kappa, w.rtol)
    # manufactured solution: ||x - x*|| / ||x*|| <= kappa * rtol
    err = np.linalg.norm(out["x"] - w.x_star) / np.linalg.norm(w.x_star)
    assert err <= kappa * w.rtol, err


def pin_history_matches_true_residual(lib):
    # the recursive residual history equals ||b - A x_k|| / ||b|| of the iterate after k steps
    A = diffusion_dirichlet(12, np.random.default_rng(3).lognormal(0, 1.0, 2 * 12 * 13))
    D = A.dense()
    b = np.random.default_rng(4).standard_normal(A.n)
    nb = np.linalg.norm(b)
    for precond in (0, 1):
        full = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=12, precond=precond, history=True,
                         lib=lib)
        assert full["history"][0] == 1.0
        for k in [1, 2, 5, 12]:
            part = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=k, precond=precond, lib=lib)
            assert part["status"] == 1 and part["iters"] == k
            true_rel = np.linalg.norm(b - D @ part["x"]) / nb
            assert abs(true_rel - full["history"][k]) <= 1e-10 * max(true_rel, 1e-3), (precond, k)
            assert part["rel_res"] == full["history"][k]


def pin_x0_restart(lib):
    A = poisson_5pt(10)
    b = np.random.default_rng(8).standard_normal(A.n)
    D = A.dense()
    xs = np.linalg.solve(D, b)
    first = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=7, lib=lib)
    rest = oracle.cg(A.row_ptr, A.col_idx, A.values, b, x0=first["x"], rtol=1e-12, maxit=1000, lib=lib)
    assert rest["status"] == 0
    assert np.linalg.norm(rest["x"] - xs) / np.linalg.norm(xs) < 1e-9
    # starting at the exact solution: 0 iterations
    at = oracle.cg(A.row_ptr, A.col_idx, A.values, D @ xs, x0=xs, rtol=1e-8, maxit=10, lib=lib)
    assert at["iters"] == 0 and at["status"] == 0


def pin_jacobi_constant_diagonal(lib):
    A = poisson_5pt(20)
    b = np.random.default_rng(9).standard_normal(A.n)
    a = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=5000, precond=0, history=True, lib=lib)
    j = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=5000, precond=1, history=True, lib=lib)
    assert a["iters"] == j["iters"]
    assert np.array_equal(a["x"], j["x"])
    assert np.array_equal(a["history"], j["history"])


def pin_jacobi_equals_scaled_cg(lib):
    # Jacobi PCG on (A, b) produces, step for step, x_k = D^{-1/2} y_k where y_k are the plain CG
    # iterates on the symmetrically scaled system (D^{-1/2} A D^{-1/2}) y = D^{-1/2} b (exact algebra;
    # agreement up to rounding).
    A = diffusion_dirichlet(10, np.random.default_rng(61).lognormal(0, 1.0, 2 * 10 * 11))
    b = np.random.default_rng(62).standard_normal(A.n)
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    d = A.dense().diagonal()
    s = 1.0 / np.sqrt(d)
    vals_scaled = A.values * s[rows] * s[A.col_idx]
    for k in [1, 2, 3, 6, 15]:
        pc = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=k, precond=1, lib=lib)
        sc = oracle.cg(A.row_ptr, A.col_idx, vals_scaled, s * b, rtol=0.0, maxit=k, precond=0, lib=lib)
        x_from_scaled = s * sc["x"]
        err = np.linalg.norm(pc["x"] - x_from_scaled) / np.linalg.norm(x_from_scaled)
        assert err <= 1e-11, (k, err)


def pin_status_codes(lib):
    A = poisson_5pt(6)
    n = A.n
    b = np.random.default_rng(1).standard_normal(n)
    z = oracle.cg(A.row_ptr, A.col_idx, A.values, np.zeros(n), x0=np.ones(n), rtol=1e-8, maxit=10, lib=lib)
    assert z["status"] == 0 and z["iters"] == 0 and not z["x"].any()
    m0 = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-8, maxit=0, lib=lib)
    assert m0["status"] == 1 and m0["iters"] == 0 and not m0["x"].any()
    neg = oracle.cg(A.row_ptr, A.col_idx, -A.values, b, rtol=1e-8, maxit=10, lib=lib)
    assert neg["status"] == 2 and neg["iters"] == 0
    bn = b.copy(); bn[3] = np.nan
    assert oracle.cg(A.row_ptr, A.col_idx, A.values, bn, rtol=1e-8, maxit=10, lib=lib)["status"] == 5
    vn = A.values.copy(); vn[7] = np.inf
    assert oracle.cg(A.row_ptr, A.col_idx, vn, b, rtol=1e-8, maxit=10, lib=lib)["status"] == 5
    vz = A.values.copy(); vz[0] = 0.0   # row 0's diagonal is its first stored entry
    assert A.col_idx[0] == 0
    assert oracle.cg(A.row_ptr, A.col_idx, vz, b, rtol=1e-8, maxit=10, precond=1, lib=lib)["status"] == 2
    # a non-finite diagonal anywhere outranks a non-positive one earlier in the matrix
    dpos = [k for k in range(int(A.row_ptr[A.n - 1]), int(A.row_ptr[A.n])) if A.col_idx[k] == A.n - 1][0]
    vb = vz.copy(); vb[dpos] = np.nan
    assert oracle.cg(A.row_ptr, A.col_idx, vb, b, rtol=1e-8, maxit=10, precond=1, lib=lib)["status"] == 5
    nc = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-12, maxit=3, lib=lib)
    assert nc["status"] == 1 and nc["iters"] == 3


# --------------------------------------------------------------------------- adjoint

def _dense_L(D, b, g):
    return float(g @ np.linalg.solve(D, b))


def pin_adjoint_identity(lib):
    A = diffusion_dirichlet(11, np.random.default_rng(21).lognormal(0, 1.0, 2 * 11 * 12))
    rng = np.random.default_rng(22)
    g, c = rng.standard_normal(A.n), rng.standard_normal(A.n)
    for precond in (0, 1):
        lam = oracle.cg(A.row_ptr, A.col_idx, A.values, g, rtol=1e-13, maxit=10000, precond=precond, lib=lib)["x"]
        y = oracle.cg(A.row_ptr, A.col_idx, A.values, c, rtol=1e-13, maxit=10000, precond=precond, lib=lib)["x"]
        lhs, rhs = float(g @ y), float(lam @ c)
        assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + abs(rhs)), (lhs, rhs)


def pin_adjoint_fd(lib):
    A = diffusion_interior(4, np.random.default_rng(31).lognormal(0, 0.5, 2 * 4 * 3), 0.01)
    D = A.dense()
    rng = np.random.default_rng(32)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    fw = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-14, maxit=10000, lib=lib)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, fw["x"], g, rtol=1e-14, maxit=10000, lib=lib)
    assert adj["status"] == 0
    # d/db_i by central differences
    for i in [0, 5, A.n - 1]:
        h = 1e-6 * max(1.0, abs(b[i]))
        bp, bm = b.copy(), b.copy()
        bp[i] += h; bm[i] -= h
        fd = (_dense_L(D, bp, g) - _dense_L(D, bm, g)) / (2 * h)
        assert abs(fd - adj["grad_b"][i]) <= 1e-7 * max(1.0, abs(fd)), (i, fd, adj["grad_b"][i])
    # d/dvalues_k: perturb one stored entry only (the perturbed matrix is not symmetric)
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    for k in [0, 1, 7, A.nnz // 2, A.nnz - 1]:
        i, j = rows[k], A.col_idx[k]
        h = 1e-6 * max(1.0, abs(A.values[k]))
        Dp, Dm = D.copy(), D.copy()
        Dp[i, j] += h; Dm[i, j] -= h
        fd = (_dense_L(Dp, b, g) - _dense_L(Dm, b, g)) / (2 * h)
        assert abs(fd - adj["grad_values"][k]) <= 1e-7 * max(1.0, abs(fd)), (k, fd, adj["grad_values"][k])


def pin_adjoint_config1_loss(lib):
    # config-1 loss L = 0.5 ||x - x_t||^2, so g = x - x_t; check a few gradient entries by FD (small grid)
    A = poisson_5pt(6)
    D = A.dense()
    rng = np.random.default_rng(41)
    x_star = rng.uniform(-1, 1, A.n)
    b = D @ x_star
    x_t = rng.uniform(-1, 1, A.n)
    fw = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-14, maxit=1000, lib=lib)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, fw["x"], fw["x"] - x_t, rtol=1e-14, maxit=1000,
                            lib=lib)

    def L(Dm, bm):
        x = np.linalg.solve(Dm, bm)
        return 0.5 * float((x - x_t) @ (x - x_t))

    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    for k in [3, 50, A.nnz - 2]:
        i, j = rows[k], A.col_idx[k]
        h = 1e-6
        Dp, Dm = D.copy(), D.copy()
        Dp[i, j] += h; Dm[i, j] -= h
        fd = (L(Dp, b) - L(Dm, b)) / (2 * h)
        assert abs(fd - adj["grad_values"][k]) <= 1e-7 * max(1.0, abs(fd))
    for i in [0, 17]:
        bp, bm = b.copy(), b.copy()
        bp[i] += 1e-6; bm[i] -= 1e-6
        fd = (L(D, bp) - L(D, bm)) / 2e-6
        assert abs(fd - adj["grad_b"][i]) <= 1e-7 * max(1.0, abs(fd))


def pin_adjoint_invariants(lib):
    A = diffusion_dirichlet(16, np.random.default_rng(51).lognormal(0, 1.0, 2 * 16 * 17))
    rng = np.random.default_rng(52)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    fw = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-13, maxit=10000, precond=1, lib=lib)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, fw["x"], g, rtol=1e-13, maxit=10000, precond=1,
                            lib=lib)
    gx = float(g @ fw["x"])
    s1 = float(adj["grad_values"] @ A.values)
    s2 = float(adj["grad_b"] @ b)
    assert abs(s1 + gx) <= 1e-9 * abs(gx), (s1, gx)
    assert abs(s2 - gx) <= 1e-9 * abs(gx), (s2, gx)
    # pattern: one gradient per stored entry, and -lambda_i x_j exactly on a hand-picked entry
    assert adj["grad_values"].shape == (A.nnz,)
    k = 5
    i = int(np.searchsorted(A.row_ptr, k, side="right") - 1)
    assert adj["grad_values"][k] == -(adj["grad_b"][i] * fw["x"][A.col_idx[k]])


def pin_adjoint_zero_gradient(lib):
    A = poisson_5pt(5)
    x = np.random.default_rng(3).standard_normal(A.n)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, x, np.zeros(A.n), rtol=1e-8, maxit=10, lib=lib)
    assert adj["status"] == 0 and adj["iters"] == 0
    assert not adj["grad_b"].any() and not adj["grad_values"].any()


# --------------------------------------------------------------------------- eigenvalue problems

def poisson_fundamental(m: int):
    """Smallest eigenvalue 4 - 4cos(pi/(m+1)) of the five-point Laplacian and its unit eigenvector,
    sin(pi (a+1)/(m+1)) sin(pi (b+1)/(m+1)) at grid point (a, b)."""
    th = np.pi / (m + 1)
    s = np.sin(th * np.arange(1, m + 1))
    v = np.outer(s, s).reshape(-1)
    return 4.0 - 4.0 * np.cos(th), v / np.linalg.norm(v)


def _eigs_general(D: np.ndarray) -> np.ndarray:
    """Eigenvalues of a (possibly non-symmetric) dense matrix, real parts ascending."""
    return np.sort(np.linalg.eigvals(D).real)


def _entry_fd(D, i, j, which, weights, h=1e-6):
    """Central difference of sum_s w_s mu_s (mu ascending) for a perturbation of the single entry (i, j)."""
    Dp, Dm = D.copy(), D.copy()
    Dp[i, j] += h
    Dm[i, j] -= h
    ep, em = _eigs_general(Dp), _eigs_general(Dm)
    return sum(w * (ep[s] - em[s]) for s, w in zip(which, weights)) / (2.0 * h)


def pin_eig_smallest_closed_form(lib):
    for m in [4, 9, 16]:
        A = poisson_5pt(m)
        mu, V = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values)
        mu0, v0 = poisson_fundamental(m)
        assert abs(mu[0] - mu0) <= 1e-13, (m, mu[0], mu0)
        assert np.max(np.abs(V[0] - v0)) <= 1e-12, m  # the fundamental mode is positive: no sign flip


def pin_eig_grad_fd(lib):
    # Hellmann-Feynman against central differences of the smallest eigenvalue, one stored entry
    # perturbed at a time (the perturbed matrix is not symmetric, so its eigenvalues are taken
    # by the general eigensolver)
    # (a random graph Laplacian plus a shift would often be disconnected, with a repeated smallest
    # eigenvalue; the Dirichlet diffusion operator's is simple)
    A = diffusion_dirichlet(5, np.random.default_rng(1).lognormal(0.0, 0.5, 2 * 5 * 6))
    D = oracle.dense(A.row_ptr, A.col_idx, A.values)
    mu, V = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 2)
    assert mu[1] - mu[0] > 0.5  # a simple eigenvalue
    gv = oracle.eig_grad_values(A.row_ptr, A.col_idx, V[:1], lib=lib)
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr))
    off = np.flatnonzero(rows != A.col_idx)
    picks = [0, int(off[0]), int(off[len(off) // 2]), A.nnz - 1, int(np.argmax(np.abs(gv)))]
    for e in picks:
        fd = _entry_fd(D, rows[e], A.col_idx[e], [0], [1.0])
        assert abs(fd - gv[e]) <= 1e-7, (e, fd, gv[e])


def pin_eig_grad_weighted_fd(lib):
    # L = 2 mu_0 - 0.5 mu_1: weights and the second eigenvector enter
    A = diffusion_dirichlet(5, np.random.default_rng(2).lognormal(0.0, 0.7, 2 * 5 * 6))
    D = oracle.dense(A.row_ptr, A.col_idx, A.values)
    mu, V = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 3)
    assert min(mu[1] - mu[0], mu[2] - mu[1]) > 0.2
    w = [2.0, -0.5]
    gv = oracle.eig_grad_values(A.row_ptr, A.col_idx, V[:2], w, lib=lib)
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr))
    for e in [1, A.nnz // 3, int(np.argmax(np.abs(gv))), int(np.argmin(gv))]:
        fd = _entry_fd(D, rows[e], A.col_idx[e], [0, 1], w)
        assert abs(fd - gv[e]) <= 1e-7, (e, fd, gv[e])


def pin_eig_grad_rayleigh_identity(lib):
    # sum_e gv_e A_e = sum_s w_s v_s^T A v_s = sum_s w_s mu_s (exact identity up to rounding), and
    # with no eigenvector the gradient is zero
    A = diffusion_dirichlet(7, np.random.default_rng(4).lognormal(0.0, 0.5, 2 * 7 * 8))
    mu, V = oracle.eig_smallest(A.row_ptr, A.col_idx, A.values, 3)
    w = np.array([1.0, -3.0, 0.25])
    gv = oracle.eig_grad_values(A.row_ptr, A.col_idx, V, w, lib=lib)
    assert abs(float(gv @ A.values) - float(w @ mu)) <= 1e-12 * float(np.abs(w) @ np.abs(mu))
    gv1 = oracle.eig_grad_values(A.row_ptr, A.col_idx, V[:1], lib=lib)
    assert abs(float(gv1 @ A.values) - mu[0]) <= 1e-13
    assert not oracle.eig_grad_values(A.row_ptr, A.col_idx, np.zeros((0, A.n)), lib=lib).any()


# --------------------------------------------------------------------------- BiCGStab (general A)

def _nonsym_dominant(n, seed):
    """A random non-symmetric CSR matrix with every row's diagonal 1 + the row's absolute sum:
    strictly diagonally dominant, so nonsingular, and far from symmetric."""
    rp, ci, v = _random_csr(n, 6, seed)
    D = _dense(rp, ci, v, n)
    D += np.diag(np.abs(D).sum(axis=1) + 1.0 - np.diag(D))
    rows, cols = np.nonzero(D)
    order = np.lexsort((cols, rows))
    rows, cols = rows[order], cols[order]
    rp2 = np.concatenate([[0], np.cumsum(np.bincount(rows, minlength=n))]).astype(np.int64)
    return rp2, cols.astype(np.int32), D[rows, cols]


def pin_transpose_dense(lib):
    rp, ci, v = _nonsym_dominant(37, 3)
    trp, tci, tv = oracle.transpose(rp, ci, v, lib=lib)
    assert np.array_equal(_dense(trp, tci, tv, 37), _dense(rp, ci, v, 37).T)
    for c in range(37):  # each column's entries in increasing row order
        assert np.all(np.diff(tci[trp[c]:trp[c + 1]]) > 0)


def pin_bicgstab_vs_dense(lib):
    cd = convection_diffusion(9, 0.6, -0.3)
    cases = [(cd.row_ptr, cd.col_idx, cd.values, cd.n), (*_nonsym_dominant(60, 5), 60)]
    for rp, ci, v, n in cases:
        D = _dense(np.asarray(rp, dtype=np.int64), ci, v, n)
        assert not np.allclose(D, D.T)
        b = np.random.default_rng(n).standard_normal(n)
        r = oracle.bicgstab(rp, ci, v, b, rtol=1e-13, maxit=1000, history=True, lib=lib)
        xd = np.linalg.solve(D, b)
        assert r["status"] == 0 and r["iters"] > 1
        assert np.linalg.norm(r["x"] - xd) <= 1e-10 * np.linalg.norm(xd)
        true_res = np.linalg.norm(b - D @ r["x"]) / np.linalg.norm(b)
        assert true_res <= 1e-12 and r["rel_res"] <= 1e-13
        assert r["history"][0] == 1.0 and abs(r["history"][-1] - r["rel_res"]) == 0.0


def pin_bicgstab_equals_cg_on_spd(lib):
    A = diffusion_dirichlet(8, np.random.default_rng(6).lognormal(0.0, 0.5, 2 * 8 * 9))
    b = np.random.default_rng(7).standard_normal(A.n)
    rb = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=1e-13, lib=lib)
    rc = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-13, lib=lib)
    assert rb["status"] == rc["status"] == 0
    assert np.linalg.norm(rb["x"] - rc["x"]) <= 1e-10 * np.linalg.norm(rc["x"])


def pin_bicgstab_adjoint_fd(lib):
    # L = g . x(A, b) for a non-symmetric A: grad_b = lambda with A^T lambda = g (so g.x = lambda.b),
    # grad_values = -lambda_i x_j, each against central differences of the dense solve
    rp, ci, v = _nonsym_dominant(30, 8)
    n = 30
    D = _dense(rp, ci, v, n)
    rng = np.random.default_rng(9)
    b, g = rng.standard_normal(n), rng.standard_normal(n)
    x = oracle.bicgstab(rp, ci, v, b, rtol=1e-14, lib=lib)["x"]
    adj = oracle.bicgstab_adjoint(rp, ci, v, x, g, rtol=1e-14, lib=lib)
    assert adj["status"] == 0
    lam = adj["grad_b"]
    assert abs(g @ x - lam @ b) <= 1e-12 * (np.abs(g) @ np.abs(x))
    assert np.linalg.norm(D.T @ lam - g) <= 1e-12 * np.linalg.norm(g)
    L = lambda DD, bb: g @ np.linalg.solve(DD, bb)  # noqa: E731
    h = 1e-6
    for k in (0, 11, 29):
        e = np.zeros(n)
        e[k] = h
        assert abs((L(D, b + e) - L(D, b - e)) / (2 * h) - lam[k]) <= 1e-7
    rows = np.repeat(np.arange(n), np.diff(rp))
    for q in (0, len(ci) // 2, len(ci) - 1, int(np.argmax(np.abs(adj["grad_values"])))):
        E = np.zeros((n, n))
        E[rows[q], ci[q]] = h
        fd = (L(D + E, b) - L(D - E, b)) / (2 * h)
        assert abs(fd - adj["grad_values"][q]) <= 1e-7, (q, fd, adj["grad_values"][q])


def pin_bicgstab_finite_termination(lib):
    # A diagonalisable non-symmetric matrix with three distinct eigenvalues: BiCG's polynomial
    # reaches the minimal polynomial at degree 3 and BiCGStab's residual carries it as a factor,
    # so in exact arithmetic the third iteration gives r = 0 (here: below 1e-9 relative)
    rng = np.random.default_rng(11)
    n = 12
    S = np.eye(n) + 0.3 * rng.standard_normal((n, n))
    D = S @ np.diag(np.repeat([1.0, 2.0, 3.0], 4)) @ np.linalg.inv(S)
    rp = np.arange(0, n * n + 1, n, dtype=np.int64)
    ci = np.tile(np.arange(n, dtype=np.int32), n)
    for seed in range(3):
        b = np.random.default_rng(seed).standard_normal(n)
        r = oracle.bicgstab(rp, ci, D.reshape(-1), b, rtol=1e-9, maxit=50, lib=lib)
        assert r["status"] == 0 and r["iters"] == 3, r["iters"]


def pin_bicgstab_status(lib):
    cd = convection_diffusion(6)
    rp, ci, v = cd.row_ptr, cd.col_idx, cd.values
    r = oracle.bicgstab(rp, ci, v, np.zeros(cd.n), lib=lib)
    assert r["status"] == 0 and r["iters"] == 0 and not r["x"].any()
    b = np.random.default_rng(2).standard_normal(cd.n)
    r = oracle.bicgstab(rp, ci, v, b, maxit=0, lib=lib)
    assert r["status"] == 1 and r["iters"] == 0 and not r["x"].any()
    xs = np.linalg.solve(_dense(np.asarray(rp, dtype=np.int64), ci, v, cd.n), b)
    r = oracle.bicgstab(rp, ci, v, b, x0=xs, rtol=1e-8, lib=lib)  # started at the solution
    assert r["status"] == 0 and r["iters"] == 0 and np.array_equal(r["x"], xs)


ALL_PINS = [
    pin_spmv_dense, pin_spmv_exact_integers, pin_dot, pin_spmv_transpose_dense, pin_matvec_grad_values,
    pin_cg_vs_dense, pin_cg_several_chunks_true_residual, pin_cg_exact_rational, pin_finite_termination, pin_eigen_closed_form_and_bound,
    pin_history_matches_true_residual, pin_x0_restart, pin_jacobi_constant_diagonal, pin_jacobi_equals_scaled_cg,
    pin_status_codes,
    pin_adjoint_identity, pin_adjoint_fd, pin_adjoint_config1_loss, pin_adjoint_invariants,
    pin_adjoint_zero_gradient,
    pin_eig_smallest_closed_form, pin_eig_grad_fd, pin_eig_grad_weighted_fd, pin_eig_grad_rayleigh_identity,
    pin_transpose_dense, pin_bicgstab_vs_dense, pin_bicgstab_equals_cg_on_spd, pin_bicgstab_adjoint_fd,
    pin_bicgstab_finite_termination, pin_bicgstab_status,
]
