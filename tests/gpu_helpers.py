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
HIST_TOL = 1e-8         # residual history, relative, first 50 iterations
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


def check_history(h_gpu, h_orc, k=50, tol=HIST_TOL):
    m = min(k + 1, len(h_gpu), len(h_orc))
    hg, ho = np.asarray(h_gpu[:m]), np.asarray(h_orc[:m])
    err = np.max(np.abs(hg - ho) / np.maximum(np.abs(ho), 1e-300))
    assert err <= tol, f"residual history differs: max rel {err:.3e} over {m} entries"
