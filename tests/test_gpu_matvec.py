"""The autograd-aware product y = A x on the GPU against the oracle (torch-sla summary,
Methodology 1: ".matvec" is differentiable; its value gradient lives on the pattern).

Values are not symmetric (the pattern is): grad_x = A^T gy goes through sla_spmv_transpose, which
gathers a_ij from row i by binary search; grad_values = gy_i x_j is one rounded product per entry,
so it is compared exactly (for float data the oracle's fp64 product of two floats, rounded once).
"""
import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, t, spmv_bound
from workloads import random_spd, poisson_5pt

pytestmark = pytest.mark.gpu


def _nonsym_values(A, seed):
    # the pattern of A (structurally symmetric) with independent random values
    return np.random.default_rng(seed).standard_normal(A.nnz)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("rowptr64", [False, True])
def test_matvec_forward_backward(dtype, rowptr64):
    A = random_spd(3000, 5.0, 7, long_rows=3)
    rp = A.row_ptr.astype(np.int64 if rowptr64 else np.int32)
    v = _nonsym_values(A, 8).astype(dtype)
    rng = np.random.default_rng(9)
    x, gy = rng.standard_normal(A.n).astype(dtype), rng.standard_normal(A.n).astype(dtype)
    dA = sla.CSRMatrix.from_numpy(rp, A.col_idx, v, "cuda:0")
    vals = dA.values.clone().requires_grad_(True)
    xt = t(x).requires_grad_(True)
    y = sla.MatVec.apply(dA.row_ptr, dA.col_idx, vals, xt)
    y.backward(t(gy))
    v64, x64, g64 = v.astype(np.float64), x.astype(np.float64), gy.astype(np.float64)
    eps = np.finfo(dtype).eps
    y_ref = oracle.spmv(A.row_ptr, A.col_idx, v64, x64)
    assert np.all(np.abs(y.detach().cpu().numpy() - y_ref) <= spmv_bound(A, x64, eps) * 4 + 4 * eps * np.abs(y_ref))
    gx_ref = oracle.spmv_transpose(A.row_ptr, A.col_idx, v64, g64)
    # the transposed product's rounding bound: 2 * len * eps * sum |a_ij gy_i| per output
    AT_abs = oracle.spmv_transpose(A.row_ptr, A.col_idx, np.abs(v64), np.abs(g64))
    lens = np.diff(A.row_ptr.astype(np.int64))
    bound = 4 * np.maximum(lens, 1) * eps * AT_abs + 4 * eps * np.abs(gx_ref) + 1e-300
    assert np.all(np.abs(xt.grad.cpu().numpy() - gx_ref) <= bound)
    gv_ref = oracle.matvec_grad_values(A.row_ptr, A.col_idx, g64, x64).astype(dtype)
    assert np.array_equal(vals.grad.cpu().numpy(), gv_ref)


def test_matvec_gradients_through_a_loss():
    # L = 0.5 ||A x - c||^2: dL/dx = A^T (A x - c), dL/dA_ij = (A x - c)_i x_j
    A = poisson_5pt(40)
    v = _nonsym_values(A, 3)
    rng = np.random.default_rng(4)
    x, c = rng.standard_normal(A.n), rng.standard_normal(A.n)
    dA = sla.CSRMatrix.from_numpy(A.row_ptr, A.col_idx, v, "cuda:0")
    vals = dA.values.clone().requires_grad_(True)
    xt = t(x).requires_grad_(True)
    loss = 0.5 * ((sla.matvec(sla.CSRMatrix(dA.row_ptr, dA.col_idx, vals), xt) - t(c)) ** 2).sum()
    loss.backward()
    r = oracle.spmv(A.row_ptr, A.col_idx, v, x) - c
    gx = oracle.spmv_transpose(A.row_ptr, A.col_idx, v, r)
    gv = oracle.matvec_grad_values(A.row_ptr, A.col_idx, r, x)
    assert np.linalg.norm(xt.grad.cpu().numpy() - gx) <= 1e-13 * np.linalg.norm(gx)
    assert np.linalg.norm(vals.grad.cpu().numpy() - gv) <= 1e-13 * np.linalg.norm(gv)


def test_spmv_transpose_refuses_a_nonsymmetric_pattern():
    # row 0 stores (0, 5) but row 5 has no (5, 0)
    n = 8
    rp = np.array([0, 2, 3, 4, 5, 6, 7, 8, 9], dtype=np.int32)
    ci = np.array([0, 5, 1, 2, 3, 4, 5, 6, 7], dtype=np.int32)
    dA = sla.CSRMatrix.from_numpy(rp, ci, np.ones(9), "cuda:0")
    with pytest.raises(sla.SlaError):
        sla.sla_spmv_transpose(dA, t(np.ones(n)))
