"""Shared helpers of the GPU parity tests: upload a workload, run libsla and the oracle, compare."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import differentiable_sparse_iterative_gb300 as sla  # noqa: E402
import oracle  # noqa: E402

# Tolerances: the fp64 and fp32 bars of the parity contract, and the iteration-count slack.
X_TOL_F64 = 1e-9        # solution, relative L2
GRAD_TOL_F64 = 1e-7     # grad_b and grad_values, relative L2
HIST_TOL = 1e-8         # residual history, relative, first 50 iterations ...
HIST_FLOOR = 1e-13      # ... with an absolute floor (in units of ||b||) for entries at rounding level
TOL_F32 = 1e-4          # float32 data, relative L2 per system
ITER_SLACK_F64 = 1      # stopping-iteration jitter near the threshold
ITER_SLACK_F32 = 0.06   # float32 CG loses orthogonality a little sooner (relative)

DEV = "cuda:0"


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def to_dev(A, dtype=None):
    vals = A.values if dtype is None else A.values.astype(dtype)
    return sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, vals, DEV)


def t(x, dtype=None):
    arr = np.asarray(x) if dtype is None else np.asarray(x).astype(dtype)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(DEV)


def spmv_bound(A, x, eps):
    """Per-row rounding bound of a row sum of len terms: 2 * len * eps * sum |a_ij x_j|."""
    rp = A.row_ptr.astype(np.int64)
    lens = np.diff(rp)
    rows = np.repeat(np.arange(A.n), lens)
    absx = np.abs(np.asarray(x, dtype=np.float64))
    s = np.zeros(A.n)
    np.add.at(s, rows, np.abs(A.values.astype(np.float64)) * absx[A.col_idx])
    return 2.0 * np.maximum(lens, 1) * eps * s + 1e-300


def check_history(h_gpu, h_orc, k=50, tol=HIST_TOL, floor=HIST_FLOOR):
    """|h_gpu - h_orc| <= tol * h_orc + floor over the first k+1 entries.

    The floor covers entries that have reached rounding level (a residual of ~1e-16 ||b||
    has no relative accuracy in either implementation)."""
    m = min(k + 1, len(h_gpu), len(h_orc))
    hg, ho = np.asarray(h_gpu[:m]), np.asarray(h_orc[:m])
    excess = np.abs(hg - ho) - (tol * np.abs(ho) + floor)
    assert np.all(excess <= 0), (f"residual history differs over {m} entries: max rel "
                                 f"{np.max(np.abs(hg - ho) / np.maximum(np.abs(ho), 1e-300)):.3e}")


def rounding_sensitivity(A, b, precond, rtol, maxit, k=50, trials=3, tol=1e-10):
    """How far the oracle's own CG trajectory survives rounding-level perturbations of b.

    Each trial moves every entry of b by one ulp (up or down at random) and reruns the oracle.
    Returns (horizon, iter_spread): horizon = first iteration where some trial's residual
    history departs from the unperturbed one by more than tol relative (k+1 if none within k);
    iter_spread = largest change of the converged iteration count.  On well-conditioned
    problems (the five-point Poisson systems, Jacobi-preconditioned diffusion) the horizon is
    past 50; on small unpreconditioned strongly variable-coefficient matrices CG's residual
    recurrence amplifies rounding within 10-30 iterations, and two correct fp64
    implementations that differ only in summation order part ways there too.
    """
    rng = np.random.default_rng(12345)
    base = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=rtol, maxit=maxit, precond=precond, history=True)
    h0 = base["history"]
    horizon, spread = k + 1, 0
    for _ in range(trials):
        up = rng.random(b.shape[0]) < 0.5
        bp = np.where(up, np.nextafter(b, np.inf), np.nextafter(b, -np.inf))
        pr = oracle.cg(A.row_ptr, A.col_idx, A.values, bp, rtol=rtol, maxit=maxit, precond=precond, history=True)
        h1 = pr["history"]
        m = min(k + 1, len(h0), len(h1))
        bad = np.nonzero(np.abs(h1[:m] - h0[:m]) > tol * np.abs(h0[:m]) + HIST_FLOOR)[0]
        if bad.size:
            horizon = min(horizon, int(bad[0]))
        spread = max(spread, abs(pr["iters"] - base["iters"]))
    return horizon, spread
