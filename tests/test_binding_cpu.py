"""The Python binding refuses to compute anywhere but on a CUDA device (CPU only, no GPU needed).

The package marshals torch tensors into libsla's C calls and has no CPU or PyTorch fallback: a
CPU tensor, or a missing library, must raise before anything is computed.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import differentiable_sparse_iterative_gb300 as sla  # noqa: E402
from differentiable_sparse_iterative_gb300 import _abi, build as sla_build  # noqa: E402
from workloads import poisson_5pt  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    sla_build.build()


def _cpu_matrix():
    A = poisson_5pt(4)
    return sla.CSRMatrix(torch.from_numpy(A.row_ptr), torch.from_numpy(A.col_idx), torch.from_numpy(A.values)), A


def test_cpu_tensors_are_refused():
    dA, A = _cpu_matrix()
    x = torch.ones(A.n, dtype=torch.float64)
    for call in (lambda: sla.sla_spmv(dA, x),
                 lambda: sla.sla_cg_solve(dA, x),
                 lambda: sla.sla_cg_adjoint(dA, x, x),
                 lambda: sla.sla_grad_values(dA, x, x),
                 lambda: sla.solve(dA, x),
                 lambda: sla.sla_eig_smallest(dA),
                 lambda: sla.sla_eig_grad_values(dA, x),
                 lambda: sla.eigsh_smallest(dA)):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_eig_weight_count_checked():
    dA, A = _cpu_matrix()
    with pytest.raises(ValueError, match="one weight per eigenvector"):
        sla.sla_eig_grad_values(dA, torch.ones(2, A.n, dtype=torch.float64), weights=[1.0])


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        _abi.load(str(tmp_path / "libsla.so"))


def test_workspace_queries_need_no_gpu():
    n = 1000
    assert sla.sla_cg_workspace_bytes(n, 1, torch.float64, 0) > 4 * 8 * n
    assert sla.sla_eig_workspace_bytes(n, torch.float64) > sla.sla_cg_workspace_bytes(n, 1, torch.float64, 0)
    assert np.int64(sla.sla_eig_workspace_bytes(n, torch.float32)) % 256 == 0
