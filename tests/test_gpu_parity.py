"""libsla (CUDA, through the C ABI) against the fp64 oracle: small and ragged cases, edge cases.

Sizes span several blocks and tiles with ragged tails; every case is seeded.
"""
import numpy as np
import pytest

from gpu_helpers import (sla, oracle, torch, rel, to_dev, t, spmv_bound, check_history, rounding_sensitivity,
                         X_TOL_F64, GRAD_TOL_F64, TOL_F32, ITER_SLACK_F64, ITER_SLACK_F32)
from workloads import poisson_5pt, diffusion_dirichlet, diffusion_interior, random_spd, config1, config3

pytestmark = pytest.mark.gpu

EPS64 = np.finfo(np.float64).eps
EPS32 = np.finfo(np.float32).eps


def _cases():
    rng = np.random.default_rng(100)
    return {
        "poisson1": poisson_5pt(1),
        "poisson2": poisson_5pt(2),
        "poisson17": poisson_5pt(17),
        "poisson33_i64": poisson_5pt(33, rowptr64=True),
        "poisson90": poisson_5pt(90),
        "dirichlet45": diffusion_dirichlet(45, rng.lognormal(0, 1.0, 2 * 45 * 46)),
        "interior31": diffusion_interior(31, rng.lognormal(0, 0.5, 2 * 31 * 30), 0.01),
        "random1025": random_spd(1025, 6.0, 7, long_rows=4),
        "random3": random_spd(3, 1.0, 8),
    }


CASES = _cases()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_spmv(name, dtype):
    A = CASES[name]
    Ad = A.astype(dtype)
    x = np.random.default_rng(1).standard_normal(A.n).astype(dtype)
    y = sla.sla_spmv(to_dev(Ad), t(x)).cpu().numpy()
    yo = oracle.spmv(A.row_ptr, A.col_idx, Ad.values.astype(np.float64), x.astype(np.float64))
    eps = EPS64 if dtype == np.float64 else EPS32
    assert np.all(np.abs(y - yo) <= spmv_bound(Ad, x, eps))


def test_spmv_exact_integers():
    A = poisson_5pt(50)
    x = np.random.default_rng(2).integers(-1000, 1000, A.n).astype(np.float64)
    y = sla.sla_spmv(to_dev(A), t(x)).cpu().numpy()
    assert np.array_equal(y, oracle.spmv(A.row_ptr, A.col_idx, A.values, x))


LOOPS = {"auto": 0, "resident": 3, "graph": 2}  # auto = the cluster kernel for these sizes


@pytest.mark.parametrize("loop", list(LOOPS))
@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("precond", [0, 1])
def test_cg_and_adjoint_f64(name, precond, loop):
    A = CASES[name]
    rng = np.random.default_rng(A.n + precond)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    rtol, maxit = 1e-10, 20000
    dA = to_dev(A)
    x, info, hist = sla.sla_cg_solve(dA, t(b), rtol=rtol, maxit=maxit, precond=precond, history=True,
                                     loop=LOOPS[loop])
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit, precond=precond, history=True)
    horizon, spread = rounding_sensitivity(A, b, precond, rtol, maxit)
    assert info.status == ref["status"] == 0
    assert abs(info.iters - ref["iters"]) <= max(ITER_SLACK_F64, 2 * spread + 1)
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    h = hist.cpu().numpy()
    assert horizon >= 8, horizon
    check_history(h, ref["history"], k=min(50, horizon - 1))
    assert np.isnan(h[info.iters + 1:]).all()  # entries past iters are not written
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, t(g), rtol=rtol, maxit=maxit, precond=precond, loop=LOOPS[loop])
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=rtol, maxit=maxit, precond=precond)
    _, aspread = rounding_sensitivity(A, g, precond, rtol, maxit, k=0)
    assert ainfo.status == adj["status"] == 0
    assert abs(ainfo.iters - adj["iters"]) <= max(ITER_SLACK_F64, 2 * aspread + 1)
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert gv.shape == (A.nnz,)
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64


def test_grad_values_exact_on_given_vectors():
    # one rounded product per entry: bit-exact against the oracle given the same lambda and x
    A = random_spd(777, 5.0, 3, long_rows=2)
    rng = np.random.default_rng(4)
    lam, x = rng.standard_normal(A.n), rng.standard_normal(A.n)
    gv = sla.sla_grad_values(to_dev(A), t(lam), t(x)).cpu().numpy()
    assert np.array_equal(gv, oracle.grad_values(A.row_ptr, A.col_idx, lam, x))


def _ragged_pattern(n, seed, long_lens=(), empty_every=7, rowptr64=False, empty_span=None):
    """Rows of 0..12 entries (every empty_every-th row empty, and all rows of empty_span), plus rows of
    the given long lengths."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 13, n)
    lens[::empty_every] = 0
    if empty_span:
        lens[empty_span[0]:empty_span[1]] = 0
    for j, L in enumerate(long_lens):
        lens[(j * 997 + 11) % n] = min(L, n)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64 if rowptr64 else np.int32)
    ci = np.concatenate([np.sort(rng.choice(n, L, replace=False)) for L in lens]).astype(np.int32)
    return rp, ci


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("rowptr64", [False, True])
def test_grad_values_tiles_chunks_long_and_empty_rows(dtype, rowptr64):
    # several 1024-row tiles with a ragged last one; rows longer than an 8192-entry chunk (split
    # across chunks), exactly one chunk long, and empty rows; one rounded product per entry, so
    # the result is exact (for float data the oracle's fp64 product of two floats is exact and
    # rounds once, as the kernel's float product does)
    n = 9 * 1024 + 77
    rp, ci = _ragged_pattern(n, 11, long_lens=(9000, 8192, 8193, 3000), rowptr64=rowptr64, empty_span=(2048, 2900))
    assert np.diff(rp.astype(np.int64)).max() > 8192 and (np.diff(rp) == 0).any()
    rng = np.random.default_rng(12)
    lam, x = rng.standard_normal(n).astype(dtype), rng.standard_normal(n).astype(dtype)
    vals = np.ones(ci.shape[0], dtype)
    dA = sla.CSRMatrix.from_numpy(rp, ci, vals, "cuda:0")
    gv = sla.sla_grad_values(dA, t(lam), t(x)).cpu().numpy()
    ref = oracle.grad_values(rp, ci, lam.astype(np.float64), x.astype(np.float64)).astype(dtype)
    assert gv.dtype == dtype and np.array_equal(gv, ref)


def test_config1_manufactured_and_loss_adjoint():
    w = config1()
    dA = to_dev(w.A)
    x, info, hist = sla.sla_cg_solve(dA, t(w.b), rtol=w.rtol, maxit=w.maxit, history=True)
    ref = oracle.cg(w.A.row_ptr, w.A.col_idx, w.A.values, w.b, rtol=w.rtol, maxit=w.maxit, history=True)
    assert info.status == 0 and abs(info.iters - ref["iters"]) <= ITER_SLACK_F64
    xs = x.cpu().numpy()
    assert rel(xs, ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"])
    # L = 0.5 ||x - x_t||^2  ->  g = x - x_t
    g_gpu = x - t(w.x_target)
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, g_gpu, rtol=w.rtol, maxit=w.maxit)
    adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, w.A.values, ref["x"], ref["x"] - w.x_target, rtol=w.rtol,
                            maxit=w.maxit)
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64


@pytest.mark.parametrize("m,batch,precond", [(16, 5, 0), (24, 3, 1), (128, 64, 0)])
def test_batched_f32(m, batch, precond):
    w = config3(m=m, batch=batch)
    P = to_dev(w.A, np.float32)
    vals, b, g = t(w.values_b), t(w.b), t(w.g)
    x, infos, hist = sla.sla_cg_solve_batched(P, vals, b, rtol=w.rtol, maxit=5000, precond=precond, history=True)
    gb, gv, ainfos = sla.sla_cg_adjoint_batched(P, vals, x, g, rtol=w.rtol, maxit=5000, precond=precond)
    xs, gbs, gvs, hs = x.cpu().numpy(), gb.cpu().numpy(), gv.cpu().numpy(), hist.cpu().numpy()
    for s in range(batch):
        v64 = w.values_b[s].astype(np.float64)
        ref = oracle.cg(w.A.row_ptr, w.A.col_idx, v64, w.b[s].astype(np.float64), rtol=w.rtol, maxit=5000,
                        precond=precond, history=True)
        assert infos[s].status == ref["status"] == 0
        assert abs(infos[s].iters - ref["iters"]) <= max(1, ITER_SLACK_F32 * ref["iters"])
        assert rel(xs[s], ref["x"]) <= TOL_F32
        check_history(hs[s], ref["history"], k=10, tol=1e-4)
        # the oracle's adjoint chains from its own forward solution, as in the fp64 tests
        adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, v64, ref["x"],
                                w.g[s].astype(np.float64), rtol=w.rtol, maxit=5000, precond=precond)
        assert ainfos[s].status == 0
        assert rel(gbs[s], adj["grad_b"]) <= TOL_F32
        assert rel(gvs[s], adj["grad_values"]) <= TOL_F32


def test_batched_f64_equals_single_systems():
    # each system of a batched solve equals the single-system solve of that system (same loop driver;
    # the graph path partitions rows by batch size, so agreement there is to rounding)
    w = config3(m=20, batch=4)
    v64 = w.values_b.astype(np.float64)
    P = to_dev(w.A)
    for loop in (sla.SLA_LOOP_GRAPH, sla.SLA_LOOP_CLUSTER):
        xb, infos, _ = sla.sla_cg_solve_batched(P, t(v64), t(w.b.astype(np.float64)), rtol=1e-10, maxit=5000,
                                                loop=loop)
        for s in range(4):
            As = sla.CSRMatrix(P.row_ptr, P.col_idx, t(v64[s]))
            xs, info, _ = sla.sla_cg_solve(As, t(w.b[s].astype(np.float64)), rtol=1e-10, maxit=5000, loop=loop)
            assert info.iters == infos[s].iters
            assert rel(xb[s].cpu().numpy(), xs.cpu().numpy()) <= 1e-12


# ----------------------------------------------------------------------------- edge cases


def _solve_both(A, b, **kw):
    x, info, _ = sla.sla_cg_solve(to_dev(A), t(b), **kw)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, **kw)
    return x.cpu().numpy(), info, ref


def test_zero_rhs_gives_zero():
    A = poisson_5pt(12)
    x0 = t(np.ones(A.n))
    x, info, _ = sla.sla_cg_solve(to_dev(A), t(np.zeros(A.n)), x0=x0, rtol=1e-8, maxit=10)
    assert info.status == 0 and info.iters == 0 and not x.cpu().numpy().any()


def test_maxit_zero_and_not_converged():
    A = poisson_5pt(30)
    b = np.random.default_rng(3).standard_normal(A.n)
    x, info, ref = _solve_both(A, b, rtol=1e-8, maxit=0)
    assert info.status == ref["status"] == 1 and info.iters == 0 and not x.any()
    x, info, ref = _solve_both(A, b, rtol=1e-12, maxit=7)
    assert info.status == ref["status"] == 1 and info.iters == ref["iters"] == 7
    assert rel(x, ref["x"]) <= 1e-12


@pytest.mark.parametrize("maxit", [1, 2, 3, 8, 9, 17])
def test_fixed_iterations_any_count(maxit):
    # rtol = 0 runs exactly maxit iterations, whatever the loop body's unroll
    A = diffusion_dirichlet(20, np.random.default_rng(5).lognormal(0, 1, 2 * 20 * 21))
    b = np.random.default_rng(6).standard_normal(A.n)
    for unroll in (2, 8):
        x, info, _ = sla.sla_cg_solve(to_dev(A), t(b), rtol=0.0, maxit=maxit, unroll=unroll)
        ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=maxit)
        assert info.iters == ref["iters"] == maxit and info.status == 1
        assert rel(x.cpu().numpy(), ref["x"]) <= 1e-12


def test_breakdown_on_negative_definite():
    A = poisson_5pt(10)
    An = A.astype(np.float64)
    An.values = -A.values
    b = np.random.default_rng(1).standard_normal(A.n)
    x, info, ref = _solve_both(An, b, rtol=1e-8, maxit=50)
    assert info.status == ref["status"] == 2 and info.iters == ref["iters"] == 0


def test_nonfinite_inputs():
    A = poisson_5pt(10)
    b = np.random.default_rng(1).standard_normal(A.n)
    bn = b.copy()
    bn[5] = np.nan
    _, info, ref = _solve_both(A, bn, rtol=1e-8, maxit=50)
    assert info.status == ref["status"] == 5
    Av = A.astype(np.float64)
    Av.values = A.values.copy()
    Av.values[11] = np.inf
    _, info, ref = _solve_both(Av, b, rtol=1e-8, maxit=50)
    assert info.status == ref["status"] == 5


def test_jacobi_bad_diagonal():
    A = poisson_5pt(10)
    b = np.random.default_rng(1).standard_normal(A.n)
    Az = A.astype(np.float64)
    Az.values = A.values.copy()
    Az.values[0] = 0.0
    _, info, ref = _solve_both(Az, b, rtol=1e-8, maxit=50, precond=1)
    assert info.status == ref["status"] == 2
    dpos = [k for k in range(int(A.row_ptr[A.n - 1]), int(A.row_ptr[A.n])) if A.col_idx[k] == A.n - 1][0]
    Az.values[dpos] = np.nan
    _, info, ref = _solve_both(Az, b, rtol=1e-8, maxit=50, precond=1)
    assert info.status == ref["status"] == 5


def test_x0_restart_and_in_place():
    A = poisson_5pt(25)
    b = np.random.default_rng(9).standard_normal(A.n)
    first = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=0.0, maxit=11)
    dA = to_dev(A)
    x0 = t(first["x"])
    x, info, _ = sla.sla_cg_solve(dA, t(b), x0=x0, rtol=1e-10, maxit=5000)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, x0=first["x"], rtol=1e-10, maxit=5000)
    assert info.status == 0 and abs(info.iters - ref["iters"]) <= 1
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    # in place: x0 and x are the same buffer
    xi = t(first["x"])
    sla.sla_cg_solve(dA, t(b), x0=xi, x=xi, rtol=1e-10, maxit=5000)
    assert rel(xi.cpu().numpy(), ref["x"]) <= X_TOL_F64


def test_empty_and_single():
    A = poisson_5pt(1)
    x, info, _ = sla.sla_cg_solve(to_dev(A), t(np.array([3.0])), rtol=1e-14, maxit=10)
    assert info.iters == 1 and x.item() == 0.75


def test_validate_csr():
    A = random_spd(300, 4.0, 2, long_rows=1)
    dA = to_dev(A)
    assert sla.sla_validate_csr(dA, check_symmetric=True) == -1
    ci = A.col_idx.copy()
    k = int(A.row_ptr[40])
    ci[k], ci[k + 1] = ci[k + 1], ci[k]  # unsorted row 40
    bad = sla.CSRMatrix(dA.row_ptr, t(ci), dA.values)
    assert sla.sla_validate_csr(bad) == 40
    v = A.values.copy()
    k7 = [k for k in range(int(A.row_ptr[7]), int(A.row_ptr[8])) if A.col_idx[k] != 7][0]
    v[k7] += 1.0  # breaks symmetry between row 7 and its partner row
    assert sla.sla_validate_csr(sla.CSRMatrix(dA.row_ptr, dA.col_idx, t(v)), check_symmetric=True) in (
        7, int(A.col_idx[k7]))
    ci2 = A.col_idx.copy()
    ci2[-1] = A.n  # out of range in the last row
    assert sla.sla_validate_csr(sla.CSRMatrix(dA.row_ptr, t(ci2), dA.values)) == A.n - 1


def test_deterministic_repeat():
    A = diffusion_dirichlet(60, np.random.default_rng(7).lognormal(0, 1, 2 * 60 * 61))
    b = t(np.random.default_rng(8).standard_normal(A.n))
    dA = to_dev(A)
    x1, i1, _ = sla.sla_cg_solve(dA, b, rtol=1e-9, maxit=5000, precond=1)
    x2, i2, _ = sla.sla_cg_solve(dA, b, rtol=1e-9, maxit=5000, precond=1)
    assert i1.iters == i2.iters and torch.equal(x1, x2)


def test_no_cpu_tensors():
    A = poisson_5pt(4)
    with pytest.raises(ValueError):
        sla.sla_cg_solve(sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, A.values, "cpu"),
                         torch.zeros(A.n, dtype=torch.float64))


@pytest.mark.parametrize("precond", [0, 1])
def test_host_loop_equals_graph_loop(precond):
    # the two loop drivers run the same kernels in the same order: identical results, bit for bit
    A = diffusion_dirichlet(40, np.random.default_rng(11).lognormal(0, 1, 2 * 40 * 41))
    b = t(np.random.default_rng(12).standard_normal(A.n))
    dA = to_dev(A)
    xg, ig, hg = sla.sla_cg_solve(dA, b, rtol=1e-9, maxit=3000, precond=precond, history=True,
                                  loop=sla.SLA_LOOP_GRAPH)
    for unroll in (2, 6):
        xh, ih, hh = sla.sla_cg_solve(dA, b, rtol=1e-9, maxit=3000, precond=precond, history=True,
                                      loop=sla.SLA_LOOP_HOST, unroll=unroll)
        assert ih.iters == ig.iters and ih.status == ig.status == 0
        assert torch.equal(xh, xg) and torch.equal(hh[: ih.iters + 1], hg[: ig.iters + 1])
    gb, gv, _ = sla.sla_cg_adjoint(dA, xg, b, rtol=1e-9, maxit=3000, precond=precond, loop=sla.SLA_LOOP_HOST)
    gb2, gv2, _ = sla.sla_cg_adjoint(dA, xg, b, rtol=1e-9, maxit=3000, precond=precond, loop=sla.SLA_LOOP_GRAPH)
    assert torch.equal(gb, gb2) and torch.equal(gv, gv2)


@pytest.mark.parametrize("precond", [0, 1])
def test_graph_loop_reused_with_other_buffers(precond):
    # the graph loop is cached by shape: later solves of the same shape with other buffers (matrix,
    # right-hand side, workspace, x) and scalars (rtol, maxit) replace the cached graph's kernel
    # arguments in place.  Each result must be the host loop's, bit for bit, and the oracle's.
    A = diffusion_dirichlet(37, np.random.default_rng(31).lognormal(0, 0.5, 2 * 37 * 38))
    _, builds0, updates0 = sla.sla_graph_cache_stats()
    keep = []  # the earlier calls' buffers stay allocated, so later calls get other addresses
    for rep, rtol in enumerate((1e-8, 1e-10, 1e-9)):
        b = np.random.default_rng(60 + rep).standard_normal(A.n)
        dA, db = to_dev(A), t(b)
        ws = torch.empty(sla.sla_cg_workspace_bytes(A.n, 1, torch.float64, precond), dtype=torch.uint8,
                         device="cuda")
        maxit = 3000 + rep
        xg, ig, _ = sla.sla_cg_solve(dA, db, rtol=rtol, maxit=maxit, precond=precond, workspace=ws,
                                     loop=sla.SLA_LOOP_GRAPH)
        xh, ih, _ = sla.sla_cg_solve(dA, db, rtol=rtol, maxit=maxit, precond=precond, loop=sla.SLA_LOOP_HOST)
        assert ig.status == ih.status == 0 and ig.iters == ih.iters and torch.equal(xg, xh)
        ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit, precond=precond)
        assert abs(ig.iters - ref["iters"]) <= ITER_SLACK_F64
        assert rel(xg.cpu().numpy(), ref["x"]) <= X_TOL_F64
        keep.append((dA, db, ws, xg))
    _, builds1, updates1 = sla.sla_graph_cache_stats()
    assert builds1 - builds0 <= 1 and updates1 - updates0 >= 2


@pytest.mark.parametrize("precond", [0, 1])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_resident_matches_graph(precond, dtype):
    # the resident kernel and the streaming kernels partition rows differently (so dot products
    # round differently) but follow the same recurrences
    A = diffusion_dirichlet(120, np.random.default_rng(21).lognormal(0, 0.5, 2 * 120 * 121)).astype(dtype)
    b = np.random.default_rng(22).standard_normal(A.n).astype(dtype)
    dA = to_dev(A)
    rtol = 1e-9 if dtype == np.float64 else 1e-5
    xr, ir, hr = sla.sla_cg_solve(dA, t(b), rtol=rtol, maxit=20000, precond=precond, history=True,
                                  loop=sla.SLA_LOOP_RESIDENT)
    xg, ig, hg = sla.sla_cg_solve(dA, t(b), rtol=rtol, maxit=20000, precond=precond, history=True,
                                  loop=sla.SLA_LOOP_GRAPH)
    assert ir.status == ig.status == 0
    tol = X_TOL_F64 if dtype == np.float64 else TOL_F32
    assert abs(ir.iters - ig.iters) <= (1 if dtype == np.float64 else max(2, 0.05 * ig.iters))
    assert rel(xr.cpu().numpy(), xg.cpu().numpy()) <= tol
    check_history(hr.cpu().numpy(), hg.cpu().numpy(), k=20, tol=1e-8 if dtype == np.float64 else 1e-4)
    assert ir.kernels == 1  # the whole solve is one launch


def _largest_m(path, precond, lo, hi):
    # the largest m whose m x m five-point Poisson system AUTO still solves on `path` (one-iteration
    # probes; the answer depends on the device's SM count and shared memory)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        A = poisson_5pt(mid)
        _, info, _ = sla.sla_cg_solve(to_dev(A), t(np.ones(A.n)), rtol=1e-30, maxit=1, precond=precond)
        lo, hi = (mid, hi) if info.path == path else (lo, mid)
    return lo


def _check_fixed_iterations(A, precond, path, k=40):
    b = np.random.default_rng(A.n).standard_normal(A.n)
    x, info, hist = sla.sla_cg_solve(to_dev(A), t(b), rtol=1e-30, maxit=k, precond=precond, history=True)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-30, maxit=k, precond=precond, history=True,
                    lib=oracle.load_parallel())
    assert info.path == path and info.status == ref["status"] == 1 and info.iters == ref["iters"] == k
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"], k=k)


@pytest.mark.parametrize("precond", [0, 1])
def test_cluster_at_capacity(precond):
    # the largest system one cluster holds in shared memory (its vectors, and the CSR slice or its
    # row offsets as they fit); one grid row more goes to the resident kernel
    m = _largest_m("cluster", precond, 60, 400)
    _check_fixed_iterations(poisson_5pt(m), precond, "cluster")
    _check_fixed_iterations(poisson_5pt(m + 1), precond, "resident")


@pytest.mark.parametrize("precond", [0, 1])
def test_resident_at_capacity(precond):
    # r, p (and 1/diag) of a block's rows and their halo bitmap fill the SM's shared memory at
    # the largest resident size; one grid row more goes to the graph loop.  Both against the oracle.
    m = _largest_m("resident", precond, 900, 1700) if precond == 0 else _largest_m("resident", precond, 700, 1400)
    for mm, path in ((m, "resident"), (m + 1, "graph")):
        _check_fixed_iterations(poisson_5pt(mm), precond, path)


def test_resident_rejects_what_does_not_fit():
    w = config3(m=8, batch=2)
    P = to_dev(w.A, np.float32)
    with pytest.raises(sla.SlaError):
        sla.sla_cg_solve_batched(P, t(w.values_b), t(w.b), rtol=1e-5, maxit=100, loop=sla.SLA_LOOP_RESIDENT)


def test_tma_spmv_step_equals_plain():
    # the TMA-staged SpMV step and the plain one do the same per-row arithmetic; they run at
    # different occupancy, so the blocks (and the order of the p.q block sums) differ
    res = {}
    try:
        for variant in (sla.SLA_SPMV_TMA, sla.SLA_SPMV_PLAIN):
            sla.sla_set_spmv_variant(variant)
            out = []
            for A, pc in [(diffusion_dirichlet(300, np.random.default_rng(3).lognormal(0, 1, 2 * 300 * 301)), 1),
                          (random_spd(5000, 6.0, 4, long_rows=5), 0)]:
                dA = to_dev(A)
                b = t(np.random.default_rng(5).standard_normal(A.n))
                x, info, _ = sla.sla_cg_solve(dA, b, rtol=1e-9, maxit=4000, precond=pc, loop=sla.SLA_LOOP_GRAPH)
                assert info.status == 0
                out.append(x.cpu().numpy())
            res[variant] = np.concatenate(out)
    finally:
        sla.sla_set_spmv_variant(sla.SLA_SPMV_PLAIN)
    assert rel(res[sla.SLA_SPMV_TMA], res[sla.SLA_SPMV_PLAIN]) <= 1e-11


@pytest.mark.parametrize("precond", [0, 1])
def test_cluster_matches_graph_batched_f64(precond):
    w = config3(m=48, batch=9)
    v64 = t(w.values_b.astype(np.float64))
    b64 = t(w.b.astype(np.float64))
    P = to_dev(w.A)
    xc, ic, _ = sla.sla_cg_solve_batched(P, v64, b64, rtol=1e-10, maxit=5000, precond=precond,
                                         loop=sla.SLA_LOOP_CLUSTER)
    xg, ig, _ = sla.sla_cg_solve_batched(P, v64, b64, rtol=1e-10, maxit=5000, precond=precond,
                                         loop=sla.SLA_LOOP_GRAPH)
    for s in range(9):
        assert ic[s].status == ig[s].status == 0 and abs(ic[s].iters - ig[s].iters) <= 1
        assert rel(xc[s].cpu().numpy(), xg[s].cpu().numpy()) <= X_TOL_F64
    assert ic[0].kernels == 1  # the whole batched solve is one launch


@pytest.mark.parametrize("loop", [sla.SLA_LOOP_HOST, sla.SLA_LOOP_GRAPH, sla.SLA_LOOP_RESIDENT, sla.SLA_LOOP_CLUSTER])
@pytest.mark.parametrize("kind", ["beyond_nnz", "decreasing"])
def test_bad_row_ptr_reported_by_every_engine(loop, kind):
    # a row pointer inside a block's (or cluster CTA's) row range is corrupted; every engine skips
    # the rows it cannot trust, reads nothing outside the caller's arrays and reports SLA_BAD_CSR
    A = poisson_5pt(20)
    rp = A.row_ptr.copy()
    j = 203  # inside the rows of one block / CTA, not at a boundary
    rp[j] = A.nnz + 50 if kind == "beyond_nnz" else rp[j - 5]
    dA = to_dev(A)
    bad = sla.CSRMatrix(t(rp), dA.col_idx, dA.values)
    b = t(np.random.default_rng(3).standard_normal(A.n))
    x, info, _ = sla.sla_cg_solve(bad, b, rtol=1e-10, maxit=50, loop=loop)
    assert info.status == sla.SLA_BAD_CSR
    assert info.path == {sla.SLA_LOOP_HOST: "host", sla.SLA_LOOP_GRAPH: "graph",
                         sla.SLA_LOOP_RESIDENT: "resident", sla.SLA_LOOP_CLUSTER: "cluster"}[loop]


def test_resident_barrier_timeout_returns_status():
    # failure detection without a fault: the grid barrier waits for one arrival that never comes,
    # gives up after a short bounded wait, and the solve returns SLA_TIMEOUT; the context stays
    # usable and the next solve is exact
    import time
    A = poisson_5pt(40)
    b = t(np.random.default_rng(5).standard_normal(A.n))
    dA = to_dev(A)
    sla.sla_test_set_barrier_wait(1, 20000)
    try:
        t0 = time.time()
        _, info, _ = sla.sla_cg_solve(dA, b, rtol=1e-10, maxit=200, loop=sla.SLA_LOOP_RESIDENT)
    finally:
        sla.sla_test_set_barrier_wait(0, 0)
    assert info.status == sla.SLA_TIMEOUT and info.path == "resident"
    assert time.time() - t0 < 60
    x, info2, _ = sla.sla_cg_solve(dA, b, rtol=1e-10, maxit=2000, loop=sla.SLA_LOOP_RESIDENT)
    xg, infog, _ = sla.sla_cg_solve(dA, b, rtol=1e-10, maxit=2000, loop=sla.SLA_LOOP_GRAPH)
    assert info2.status == 0 and abs(info2.iters - infog.iters) <= 1
    assert rel(x.cpu().numpy(), xg.cpu().numpy()) <= X_TOL_F64


@pytest.mark.parametrize("m", [140, 150])
def test_batched_f32_several_row_groups(m):
    # 40 fp32 systems on 4-CTA clusters: m = 140 keeps the row offsets on chip (streamed SpMV with
    # batched entry loads), m = 150 does not fit them (plain row loop); both give each thread more
    # than 8 rows, so the fp32 partial sums go through several row groups
    batch = 40
    w = config3(m=m, batch=batch)
    P = to_dev(w.A, np.float32)
    vals, b, g = t(w.values_b), t(w.b), t(w.g)
    x, infos, _ = sla.sla_cg_solve_batched(P, vals, b, rtol=w.rtol, maxit=5000)
    gb, gv, ainfos = sla.sla_cg_adjoint_batched(P, vals, x, g, rtol=w.rtol, maxit=5000)
    assert infos[0].path == "cluster"
    xs, gbs, gvs = x.cpu().numpy(), gb.cpu().numpy(), gv.cpu().numpy()
    for s in (0, 17, batch - 1):
        v64 = w.values_b[s].astype(np.float64)
        ref = oracle.cg(w.A.row_ptr, w.A.col_idx, v64, w.b[s].astype(np.float64), rtol=w.rtol, maxit=5000)
        assert infos[s].status == ref["status"] == 0
        assert abs(infos[s].iters - ref["iters"]) <= max(1, ITER_SLACK_F32 * ref["iters"])
        assert rel(xs[s], ref["x"]) <= TOL_F32
        adj = oracle.cg_adjoint(w.A.row_ptr, w.A.col_idx, v64, ref["x"],
                                w.g[s].astype(np.float64), rtol=w.rtol, maxit=5000)
        assert ainfos[s].status == 0
        assert rel(gbs[s], adj["grad_b"]) <= TOL_F32
        assert rel(gvs[s], adj["grad_values"]) <= TOL_F32


@pytest.mark.parametrize("case", ["poisson179", "dirichlet150_jacobi"])
def test_cluster_two_p_buffers_streamed_matrix(case):
    # one fp64 system on a 16-CTA cluster whose CSR slice does not fit on chip (the SpMV streams it,
    # row offsets staged) while two p buffers do: partner rows' p_k formed from the partner's r_k
    # (1/diag) and p_{k-1}, two cluster barriers per iteration; against the oracle
    if case == "poisson179":
        A, precond = poisson_5pt(179), 0
    else:
        m = 150
        A, precond = diffusion_dirichlet(m, np.random.default_rng(8).lognormal(0, 1.0, 2 * m * (m + 1))), 1
    b = np.random.default_rng(9).standard_normal(A.n)
    g = np.random.default_rng(10).standard_normal(A.n)
    dA = to_dev(A)
    x, info, hist = sla.sla_cg_solve(dA, t(b), rtol=1e-10, maxit=20000, precond=precond, history=True,
                                     loop=sla.SLA_LOOP_CLUSTER)
    gb, gv, ainfo = sla.sla_cg_adjoint(dA, x, t(g), rtol=1e-10, maxit=20000, precond=precond,
                                       loop=sla.SLA_LOOP_CLUSTER)
    assert info.path == "cluster" and info.kernels == 1
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=20000, precond=precond, history=True)
    adj = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, ref["x"], g, rtol=1e-10, maxit=20000, precond=precond)
    assert info.status == ref["status"] == 0 and abs(info.iters - ref["iters"]) <= ITER_SLACK_F64
    assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
    check_history(hist.cpu().numpy(), ref["history"])
    assert ainfo.status == 0 and abs(ainfo.iters - adj["iters"]) <= ITER_SLACK_F64
    assert rel(gb.cpu().numpy(), adj["grad_b"]) <= GRAD_TOL_F64
    assert rel(gv.cpu().numpy(), adj["grad_values"]) <= GRAD_TOL_F64
