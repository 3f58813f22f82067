"""Input generators: sizes, structure and the closed forms the assembly must satisfy (CPU only)."""
import numpy as np
import pytest

from workloads import (poisson_5pt, diffusion_interior, diffusion_dirichlet, random_spd, config1, config3,
                       small_poisson, convection_diffusion, config_by_name)
from oracle_pins import poisson_eigs


def _canonical(A):
    rp = A.row_ptr.astype(np.int64)
    assert rp[0] == 0 and rp[-1] == A.nnz and np.all(np.diff(rp) >= 1)
    for i in range(A.n):
        cols = A.col_idx[rp[i]:rp[i + 1]]
        assert np.all(np.diff(cols) > 0) and i in cols and cols.min() >= 0 and cols.max() < A.n


@pytest.mark.parametrize("m", [1, 2, 3, 5, 16])
def test_poisson_structure(m):
    A = poisson_5pt(m)
    assert A.n == m * m and A.nnz == 5 * m * m - 4 * m
    assert A.row_ptr.dtype == np.int32 and A.col_idx.dtype == np.int32 and A.values.dtype == np.float64
    _canonical(A)
    D = A.dense()
    assert np.array_equal(D, D.T)
    if m <= 16:
        assert np.max(np.abs(np.linalg.eigvalsh(D) - np.sort(poisson_eigs(m)))) < 1e-12
    # interior rows (four neighbours) sum to zero
    a, c = np.divmod(np.arange(A.n), m)
    interior = (a > 0) & (a < m - 1) & (c > 0) & (c < m - 1)
    assert np.all(D.sum(axis=1)[interior] == 0)


def test_poisson_int64_rowptr():
    A = poisson_5pt(9, rowptr64=True)
    B = poisson_5pt(9)
    assert A.row_ptr.dtype == np.int64 and np.array_equal(A.row_ptr, B.row_ptr.astype(np.int64))


def test_dirichlet_reduces_to_poisson():
    m = 12
    A = diffusion_dirichlet(m, np.ones(2 * m * (m + 1)))
    P = poisson_5pt(m)
    assert np.array_equal(A.values, P.values) and np.array_equal(A.col_idx, P.col_idx)


def test_interior_row_sums_and_spd():
    m = 9
    k = np.random.default_rng(0).lognormal(0, 0.5, 2 * m * (m - 1))
    A = diffusion_interior(m, k, 0.01)
    _canonical(A)
    D = A.dense()
    assert np.array_equal(D, D.T)
    assert np.allclose(D.sum(axis=1), 0.01, atol=1e-12, rtol=0)
    assert np.linalg.eigvalsh(D)[0] > 0
    # first horizontal edge joins unknowns 0 and 1; first vertical edge joins 0 and m
    assert D[0, 1] == -k[0] and D[0, m] == -k[m * (m - 1)]


def test_dirichlet_edge_order():
    m = 4
    k = np.arange(1, 2 * m * (m + 1) + 1, dtype=np.float64)
    A = diffusion_dirichlet(m, k)
    D = A.dense()
    # h[0,1] (index 1) joins (0,0)-(0,1); v[1,0] (index m(m+1) + m) joins (0,0)-(1,0)
    assert D[0, 1] == -2.0 and D[0, m] == -(m * (m + 1) + m + 1)
    # diagonal of (0,0): west h[0,0] + north v[0,0] + east h[0,1] + south v[1,0]
    assert D[0, 0] == 1.0 + (m * (m + 1) + 1) + 2.0 + (m * (m + 1) + m + 1)
    assert np.linalg.eigvalsh(D)[0] > 0 and np.array_equal(D, D.T)


def test_random_spd_ragged():
    A = random_spd(300, 4.0, 1, long_rows=3)
    _canonical(A)
    lens = np.diff(A.row_ptr.astype(np.int64))
    assert lens.max() > 100 and lens.min() >= 1
    D = A.dense()
    assert np.array_equal(D, D.T) and np.linalg.eigvalsh(D)[0] > 0


def test_config1_manufactured():
    w = config1()
    assert w.A.n == 4096 and w.A.nnz == 20224
    assert np.allclose(w.A.dense() @ w.x_star, w.b, atol=1e-14, rtol=0)


def test_config3_small_batch():
    w = config3(m=8, batch=3)
    assert w.values_b.shape == (3, w.A.nnz) and w.values_b.dtype == np.float32
    assert w.b.shape == (3, 64) and w.g.shape == (3, 64) and w.b.dtype == np.float32
    # systems differ and follow their own seeds
    assert not np.array_equal(w.values_b[0], w.values_b[1])
    again = config3(m=8, batch=2)
    assert np.array_equal(again.values_b[1], w.values_b[1])


def test_small_poisson_seeded():
    a, b = small_poisson(10, 3), small_poisson(10, 3)
    assert np.array_equal(a.b, b.b) and np.array_equal(a.g, b.g)


@pytest.mark.parametrize("m", [1, 2, 6, 11])
def test_convection_diffusion_structure(m):
    # the five-point pattern of the Poisson matrix; with no convection, the Poisson matrix itself;
    # otherwise its symmetric part is the Poisson matrix and its skew part +-cx (east / west),
    # +-cy (south / north); a nonsingular M-matrix for |cx|, |cy| < 1
    cx, cy = 0.4, 0.25
    A = convection_diffusion(m, cx, cy)
    P = poisson_5pt(m)
    _canonical(A)
    assert np.array_equal(A.row_ptr, P.row_ptr) and np.array_equal(A.col_idx, P.col_idx)
    assert np.array_equal(convection_diffusion(m, 0.0, 0.0).values, P.values)
    D, DP = A.dense(), P.dense()
    assert np.allclose(0.5 * (D + D.T), DP, rtol=0, atol=1e-15)
    K = 0.5 * (D - D.T)
    i = np.arange(A.n)
    a, c = np.divmod(i, m)
    east = c < m - 1
    south = a < m - 1
    assert np.allclose(K[i[east], i[east] + 1], cx, rtol=0, atol=1e-15)
    assert np.allclose(K[i[south], i[south] + m], cy, rtol=0, atol=1e-15)
    assert np.count_nonzero(np.abs(K) > 1e-15) == 2 * (np.count_nonzero(east) + np.count_nonzero(south))
    off = D - np.diag(np.diag(D))
    assert np.all(off <= 0) and np.all(D.sum(axis=1) >= -1e-15)
    if A.n > 1:
        assert np.min(np.linalg.eigvals(D).real) > 0
    B = convection_diffusion(m, cx, cy, rowptr64=True)
    assert B.row_ptr.dtype == np.int64 and np.array_equal(B.values, A.values)


def test_convdiff_bicgstab_workload():
    w = config_by_name("convdiff1000_bicgstab", m=30)
    assert w.A.n == 900 and w.A.nnz == 5 * 900 - 4 * 30 and w.rtol == 1e-8 and w.meta["method"] == "bicgstab"
    assert np.array_equal(w.b, np.random.default_rng(0).standard_normal(900))
    assert np.array_equal(w.g, np.random.default_rng(1).standard_normal(900))
