"""BiCGStab for a general A (libsla, through the C ABI) against the fp64 oracle.

Non-symmetric inputs (residual history compared over the first 20 iterations, or up to where the
oracle parts from itself under rounding-level changes): the convection-diffusion operator on the five-point pattern (central
differences, structurally symmetric), a random diagonally dominant pattern with non-symmetric
values, and structurally non-symmetric patterns (random rows, upper bidiagonal) whose adjoint
builds A^T explicitly.  Checked: the solution at 1e-9, the iteration count, the first residual-history entries
at 1e-8, the adjoint (A^T lambda = g) gradients grad_b and grad_values at 1e-7 with the oracle's
adjoint chained from its own solution, and the status cases.
"""
import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, to_dev, t, check_history, X_TOL_F64, GRAD_TOL_F64, TOL_F32
from workloads import CSR, convection_diffusion, poisson_5pt, random_spd

pytestmark = pytest.mark.gpu


def _nonsym_random(n, seed):
    # random_spd's (symmetric) pattern with every off-diagonal value scaled by its own factor in
    # [0.6, 1): still diagonally dominant, no longer symmetric
    A = random_spd(n, 6.0, seed, long_rows=3)
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    f = np.random.default_rng(seed + 1).uniform(0.6, 1.0, A.nnz)
    v = np.where(rows == A.col_idx, A.values, A.values * f)
    return CSR(A.n, A.row_ptr, A.col_idx, v)


CASES = {
    "cd1": convection_diffusion(1),
    "cd2": convection_diffusion(2),
    "cd17": convection_diffusion(17, 0.7, -0.4),
    "cd45_i64": convection_diffusion(45, 0.3, 0.5, rowptr64=True),
    "cd120": convection_diffusion(120),
    "random1025": _nonsym_random(1025, 5),
}


LOOPS = {"resident": sla.SLA_LOOP_AUTO, "host": sla.SLA_LOOP_HOST}


def history_horizon(A, b, rtol, maxit, k=20, trials=3):
    """The first k residual-history entries, cut before the oracle parts from itself by more than the
    history bar: under one-ulp changes of b (every entry up or down at random), and between its two
    builds, which differ only in the dot products' summation order, as the GPU does.  BiCGStab
    amplifies rounding quickly on some matrices: on the random non-symmetric case one-ulp changes
    of b part the oracle from itself at iteration 9."""
    def apart(h, h0):
        m = min(len(h), len(h0), k + 1)
        idx = np.nonzero(np.abs(h[:m] - h0[:m]) > 1e-8 * np.abs(h0[:m]) + 1e-13)[0]
        return int(idx[0]) - 1 if idx.size else k

    run = lambda bb, lib=None: oracle.bicgstab(A.row_ptr, A.col_idx, A.values, bb, rtol=rtol, maxit=maxit,
                                               history=True, lib=lib)["history"]
    h0 = run(b)
    horizon = apart(run(b, oracle.load_parallel()), h0)
    for tr in range(trials):
        sgn = np.where(np.random.default_rng(200 + tr).random(A.n) < 0.5, -1.0, 1.0)
        horizon = min(horizon, apart(run(b + sgn * np.spacing(b)), h0))
    return horizon


def iteration_spread(A, b, rtol, maxit, trials=4):
    """How far the oracle's own stopping iteration moves when every entry of b moves by one ulp
    (up or down at random): BiCGStab's residual is not monotone, and near the threshold two
    correct fp64 runs that differ only in summation order can stop a few iterations apart."""
    base = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit)["iters"]
    spread = 0
    for tr in range(trials):
        sgn = np.where(np.random.default_rng(100 + tr).random(A.n) < 0.5, -1.0, 1.0)
        it = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b + sgn * np.spacing(b), rtol=rtol, maxit=maxit)["iters"]
        spread = max(spread, abs(it - base))
    return spread


@pytest.mark.parametrize("loop", list(LOOPS))
@pytest.mark.parametrize("name", list(CASES))
def test_bicgstab_and_adjoint_match_the_oracle(name, loop):
    A = CASES[name]
    rng = np.random.default_rng(A.n)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    rtol, maxit = 1e-10, 5000
    dA = to_dev(A)
    x, info, hist = sla.sla_bicgstab_solve(dA, t(b), rtol=rtol, maxit=maxit, history=True, loop=LOOPS[loop])
    assert info.path == loop
    ref = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit, history=True)
    assert info.status == ref["status"] == 0, (info, ref["status"])
    slack = 1 + max(ref["iters"] // 20, iteration_spread(A, b, rtol, maxit))
    assert abs(info.iters - ref["iters"]) <= slack, (info.iters, ref["iters"], slack)
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    h = hist.cpu().numpy()
    check_history(h, ref["history"], k=min(ref["iters"], history_horizon(A, b, rtol, maxit)))
    assert np.isnan(h[info.iters + 1:]).all()
    gb, gv, ainfo = sla.sla_bicgstab_adjoint(dA, x, t(g), rtol=rtol, maxit=maxit, loop=LOOPS[loop])
    adj = oracle.bicgstab_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=rtol, maxit=maxit)
    assert ainfo.status == adj["status"] == 0 and ainfo.path == loop
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64


@pytest.mark.parametrize("loop", list(LOOPS))
def test_bicgstab_from_a_start_vector(loop):
    # r0 = b - A x0 and rhat = r0 from a random x0, against the oracle from the same x0
    A = CASES["cd45_i64"]
    rng = np.random.default_rng(11)
    b, x0 = rng.standard_normal(A.n), rng.standard_normal(A.n)
    x, info, hist = sla.sla_bicgstab_solve(to_dev(A), t(b), x0=t(x0), rtol=1e-10, history=True, loop=LOOPS[loop])
    ref = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, x0=x0, rtol=1e-10, history=True)
    assert info.status == ref["status"] == 0 and info.path == loop
    assert abs(info.iters - ref["iters"]) <= 1 + max(ref["iters"] // 20, iteration_spread(A, b, 1e-10, 100000))
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"], k=min(8, ref["iters"]))


def test_bicgstab_on_spd_equals_the_cg_solution():
    A = poisson_5pt(40)
    b = np.random.default_rng(3).standard_normal(A.n)
    dA = to_dev(A)
    xb, ib, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-12, maxit=5000)
    xc, ic, _ = sla.sla_cg_solve(dA, t(b), rtol=1e-12, maxit=5000)
    assert ib.status == ic.status == 0
    assert rel(xb.cpu().numpy(), xc.cpu().numpy()) <= 1e-10


@pytest.mark.parametrize("loop", list(LOOPS))
def test_bicgstab_deterministic_repeat(loop):
    A = CASES["cd120"]
    dA, b = to_dev(A), t(np.random.default_rng(4).standard_normal(A.n))
    x1, i1, h1 = sla.sla_bicgstab_solve(dA, b, rtol=1e-10, history=True, loop=LOOPS[loop])
    x2, i2, h2 = sla.sla_bicgstab_solve(dA, b, rtol=1e-10, history=True, loop=LOOPS[loop])
    assert i1.iters == i2.iters and torch.equal(x1, x2) and torch.equal(h1[: i1.iters + 1], h2[: i2.iters + 1])


def test_bicgstab_engines_agree_at_1m_rows():
    # the 1M-row convection-diffusion system of the bench, resident kernel (152 chunks) and host
    # loop (band-swept tiles).  What holds at any size: each solution's true residual, recomputed in
    # fp64 on the host, meets the tolerance.  Two such solutions differ by up to cond(A) * rtol in
    # principle (cond ~ 4e5 here); they agree to ~1e-7, checked at 1e-6.
    A = convection_diffusion(1000)
    b = np.random.default_rng(0).standard_normal(A.n)
    dA = to_dev(A)
    xr, ir, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-8)
    xh, ih, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-8, loop=sla.SLA_LOOP_HOST)
    assert ir.path == "resident" and ih.path == "host"
    assert ir.status == ih.status == 0 and abs(ir.iters - ih.iters) <= 2 + ir.iters // 50
    sp = pytest.importorskip("scipy.sparse")
    M = sp.csr_matrix((A.values, A.col_idx, A.row_ptr.astype(np.int64)), shape=(A.n, A.n))
    for xx, info in ((xr, ir), (xh, ih)):
        res = np.linalg.norm(b - M @ xx.cpu().numpy()) / np.linalg.norm(b)
        assert res <= 1.05e-8 and abs(res - info.rel_res) <= 1e-3 * 1e-8, (res, info)
    assert rel(xr.cpu().numpy(), xh.cpu().numpy()) <= 1e-6
    # the adjoint at the same size: A^T lambda = g to tolerance (true residual), and grad_values is
    # -lambda_i x_j entry by entry (one rounded product: exact)
    g = np.random.default_rng(1).standard_normal(A.n)
    gb, gv, ai = sla.sla_bicgstab_adjoint(dA, xr, t(g), rtol=1e-8)
    assert ai.status == 0 and ai.path == "resident"
    lam, x_np = gb.cpu().numpy(), xr.cpu().numpy()
    assert np.linalg.norm(g - M.T @ lam) / np.linalg.norm(g) <= 1.05e-8
    rows = np.repeat(np.arange(A.n), np.diff(A.row_ptr.astype(np.int64)))
    assert np.array_equal(gv.cpu().numpy(), -(lam[rows] * x_np[A.col_idx]))


def test_bicgstab_resident_barrier_timeout_returns_status():
    # failure detection without a fault: every grid barrier waits for one arrival that never comes,
    # gives up after a short bounded wait, and the solve returns SLA_TIMEOUT; the next solve is exact
    import time
    A = CASES["cd120"]
    b = t(np.random.default_rng(5).standard_normal(A.n))
    dA = to_dev(A)
    sla.sla_test_set_barrier_wait(1, 20000)
    try:
        t0 = time.time()
        _, info, _ = sla.sla_bicgstab_solve(dA, b, rtol=1e-10, maxit=200)
    finally:
        sla.sla_test_set_barrier_wait(0, 0)
    assert info.status == sla.SLA_TIMEOUT and info.path == "resident"
    assert time.time() - t0 < 60
    x, info2, _ = sla.sla_bicgstab_solve(dA, b, rtol=1e-10)
    xh, infoh, _ = sla.sla_bicgstab_solve(dA, b, rtol=1e-10, loop=sla.SLA_LOOP_HOST)
    assert info2.status == 0 and abs(info2.iters - infoh.iters) <= 1
    assert rel(x.cpu().numpy(), xh.cpu().numpy()) <= X_TOL_F64


def test_bicgstab_autograd_node():
    A = CASES["cd17"]
    rng = np.random.default_rng(8)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    dA = to_dev(A)
    vals = dA.values.clone().requires_grad_(True)
    bt = t(b).requires_grad_(True)
    x = sla.solve(dA.with_values(vals), bt, rtol=1e-12, method="bicgstab")
    x.backward(t(g))
    xd, _, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-12)
    gbd, gvd, _ = sla.sla_bicgstab_adjoint(dA, xd, t(g), rtol=1e-12)
    assert torch.equal(x.detach(), xd) and torch.equal(bt.grad, gbd) and torch.equal(vals.grad, gvd)
    ref = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=1e-12)
    adj = oracle.bicgstab_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-12)
    assert rel(vals.grad.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64
    # method style
    x2 = dA.solve(t(b), rtol=1e-12, method="bicgstab")
    assert torch.equal(x2, xd)


def test_bicgstab_float32():
    A = convection_diffusion(40)
    b = np.random.default_rng(9).standard_normal(A.n)
    x, info, _ = sla.sla_bicgstab_solve(to_dev(A, np.float32), t(b, np.float32), rtol=1e-5)
    ref = oracle.bicgstab(A.row_ptr, A.col_idx, A.values.astype(np.float32).astype(np.float64),
                          b.astype(np.float32).astype(np.float64), rtol=1e-5)
    assert info.status == 0 and x.dtype == torch.float32
    assert rel(x.cpu().numpy(), ref["x"]) <= TOL_F32


@pytest.mark.parametrize("loop", list(LOOPS))
def test_bicgstab_status_cases(loop):
    lp = LOOPS[loop]
    A = convection_diffusion(12)
    dA = to_dev(A)
    # b = 0: x = 0 after no iteration, whatever x0
    x, info, _ = sla.sla_bicgstab_solve(dA, t(np.zeros(A.n)), x0=t(np.ones(A.n)), loop=lp)
    assert info.status == 0 and info.iters == 0 and not x.cpu().numpy().any()
    b = np.random.default_rng(1).standard_normal(A.n)
    # maxit = 0: not converged, x = x0 (0)
    x, info, _ = sla.sla_bicgstab_solve(dA, t(b), maxit=0, loop=lp)
    assert info.status == sla.SLA_NOT_CONVERGED and info.iters == 0 and not x.cpu().numpy().any()
    # started at the oracle's solution: converged before the first iteration
    xs = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=1e-14)["x"]
    x, info, _ = sla.sla_bicgstab_solve(dA, t(b), x0=t(xs), rtol=1e-8, loop=lp)
    assert info.status == 0 and info.iters == 0 and np.array_equal(x.cpu().numpy(), xs)
    # fixed iteration count, against the oracle's
    x, info, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-30, maxit=7, loop=lp)
    r = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=1e-30, maxit=7)
    assert info.status == r["status"] == sla.SLA_NOT_CONVERGED and info.iters == r["iters"] == 7
    assert rel(x.cpu().numpy(), r["x"]) <= 1e-12
    # no preconditioner option: rejected by the binding, and by the C entry point
    with pytest.raises(ValueError):
        sla.solve(dA, t(b), precond=sla.SLA_PRECOND_JACOBI, method="bicgstab")
    import ctypes
    from differentiable_sparse_iterative_gb300 import _abi, _csr_struct, _opts
    ws = torch.empty(sla.sla_bicgstab_workspace_bytes(A.n, A.nnz, torch.float64), dtype=torch.uint8,
                     device="cuda:0")
    xo = torch.empty(A.n, dtype=torch.float64, device="cuda:0")
    st = sla.lib().sla_bicgstab_solve(ctypes.byref(_csr_struct(dA)), t(b).data_ptr(), None,
                                      ctypes.byref(_opts(1e-8, 100, sla.SLA_PRECOND_JACOBI)), xo.data_ptr(),
                                      ctypes.byref(_abi.sla_cg_info()), None, ws.data_ptr(), ws.numel(),
                                      torch.cuda.current_stream().cuda_stream)
    assert st == sla.SLA_INVALID_ARG


def _nonsym_pattern(n, seed):
    """A structurally non-symmetric, strictly diagonally dominant matrix: every row its diagonal
    and 0-5 random off-diagonal columns (every 97th row 40), values U(-1, 1), the diagonal
    1 + the row's absolute off-diagonal sum."""
    rng = np.random.default_rng(seed)
    rp, ci, vals = [0], [], []
    for i in range(n):
        k = 40 if i % 97 == 0 else int(rng.integers(0, 6))
        off = rng.choice(np.delete(np.arange(n), i), size=min(k, n - 1), replace=False)
        ov = rng.uniform(-1.0, 1.0, off.size)
        cols = np.concatenate([off, [i]])
        v = np.concatenate([ov, [1.0 + np.abs(ov).sum()]])
        order = np.argsort(cols)
        ci.extend(cols[order])
        vals.extend(v[order])
        rp.append(len(ci))
    return CSR(n, np.array(rp, dtype=np.int32), np.array(ci, dtype=np.int32), np.array(vals))


@pytest.mark.parametrize("loop", list(LOOPS))
def test_bicgstab_adjoint_on_a_pattern_without_partners(loop):
    # no stored (j, i) for most (i, j): the adjoint builds A^T explicitly, as the oracle does
    A = _nonsym_pattern(3000, 4)
    rp64 = A.row_ptr.astype(np.int64)
    rows = np.repeat(np.arange(A.n), np.diff(rp64))
    assert not set(zip(rows.tolist(), A.col_idx.tolist())) <= set(zip(A.col_idx.tolist(), rows.tolist()))
    rng = np.random.default_rng(12)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    dA = to_dev(A)
    x, info, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-11, loop=LOOPS[loop])
    ref = oracle.bicgstab(A.row_ptr, A.col_idx, A.values, b, rtol=1e-11)
    assert info.status == ref["status"] == 0 and rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    gb, gv, ai = sla.sla_bicgstab_adjoint(dA, x, t(g), rtol=1e-11, loop=LOOPS[loop])
    adj = oracle.bicgstab_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-11)
    assert ai.status == adj["status"] == 0 and ai.path == loop
    assert abs(ai.iters - adj["iters"]) <= 2 + adj["iters"] // 10, (ai.iters, adj["iters"])
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64
    # the transpose's rows are sorted after the scatter: the same bits every time
    gb2, gv2, _ = sla.sla_bicgstab_adjoint(dA, x, t(g), rtol=1e-11, loop=LOOPS[loop])
    assert torch.equal(gb, gb2) and torch.equal(gv, gv2)


def test_bicgstab_adjoint_upper_bidiagonal():
    # an upper-bidiagonal pattern, (i, i+1) stored and (i+1, i) not, with random values and b.
    # (Constant values with b = ones is a degenerate case for the method itself: there rhat.r is zero
    # in exact arithmetic from the third iteration on, and the trajectory is decided by rounding.)
    n = 50
    rng = np.random.default_rng(21)
    rp = np.concatenate([[0], np.cumsum([2] * (n - 1) + [1])]).astype(np.int32)
    ci = np.concatenate([[i, i + 1] for i in range(n - 1)] + [[n - 1]]).astype(np.int32)
    diag = ci == np.repeat(np.arange(n), np.diff(rp))
    v = np.where(diag, rng.uniform(2.0, 4.0, ci.shape[0]), rng.uniform(-1.0, 1.0, ci.shape[0]))
    b = rng.standard_normal(n)
    A = CSR(n, rp, ci, v)
    dA = to_dev(A)
    x, info, _ = sla.sla_bicgstab_solve(dA, t(b), rtol=1e-12)
    assert info.status == 0
    ref = oracle.bicgstab(rp, ci, v, b, rtol=1e-12)
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    assert rel(x.cpu().numpy(), np.linalg.solve(A.dense(), b)) <= 1e-10
    gb, gv, ainfo = sla.sla_bicgstab_adjoint(dA, x, t(b), rtol=1e-12)
    adj = oracle.bicgstab_adjoint(rp, ci, v, ref["x"], b, rtol=1e-12)
    assert ainfo.status == adj["status"] == 0
    assert rel(gb.cpu().numpy(), np.linalg.solve(A.dense().T, b)) <= 1e-10
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64
    # through autograd
    vals = dA.values.clone().requires_grad_(True)
    sla.solve(dA.with_values(vals), t(b), rtol=1e-12, method="bicgstab").backward(t(b))
    assert torch.equal(vals.grad, gv)


@pytest.mark.parametrize("loop", list(LOOPS))
def test_bicgstab_reports_a_malformed_pattern(loop):
    # a column index past n: every kernel checks columns before it reads, skips the entry and
    # raises the flag; the solve and the adjoint both report SLA_BAD_CSR
    A = convection_diffusion(10)
    ci = A.col_idx.copy()
    ci[7] = A.n
    dA = sla.CSRMatrix.from_numpy(A.row_ptr, ci, A.values, "cuda:0")
    b = t(np.random.default_rng(2).standard_normal(A.n))
    x, info, _ = sla.sla_bicgstab_solve(dA, b, rtol=1e-10, loop=LOOPS[loop])
    assert info.status == sla.SLA_BAD_CSR
    _, _, ainfo = sla.sla_bicgstab_adjoint(dA, x, b, rtol=1e-10, loop=LOOPS[loop])
    assert ainfo.status == sla.SLA_BAD_CSR
