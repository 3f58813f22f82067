"""The allocation-free solve entry point (sla_cg_solve_static), called through the C ABI.

Some callers cannot allocate device memory (a plugin inside an application that owns all
device memory, a latency-critical path where allocation is not allowed, a binding with no
allocator).  sla_cg_solve_static serves them from a fixed scratch array inside the library.
This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import sla, torch, rel, to_dev, t, X_TOL_F64
from differentiable_sparse_iterative_gb300 import _abi
from workloads import diffusion_dirichlet

pytestmark = pytest.mark.gpu


def _static_solve(A, b, rtol, maxit, precond, x):
    lib = sla.lib()
    o = _abi.sla_cg_opts()
    o.rtol, o.maxit, o.precond, o.unroll, o.loop, o.reserved = rtol, maxit, precond, 0, 0, 0
    info = _abi.sla_cg_info()
    st = lib.sla_cg_solve_static(ctypes.byref(sla._csr_struct(A)), b.data_ptr(), None, ctypes.byref(o),
                                 x.data_ptr(), ctypes.byref(info), None,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, sla.sla_status_string(st)
    return info


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    m = 160  # n = 25,600 unknowns: within the 65,536 limit, several blocks and tiles
    A = diffusion_dirichlet(m, np.random.default_rng(5).lognormal(0, 1.0, 2 * m * (m + 1)))
    dA = to_dev(A)
    rng = np.random.default_rng(6)
    cases = [(t(rng.standard_normal(A.n)), 0), (t(rng.standard_normal(A.n)), 1)]
    for b, precond in cases:  # two calls in a row share the scratch array
        # the existing entry point, driven by the same kernels (the host loop) as the static one
        x_ref, info_ref, _ = sla.sla_cg_solve(dA, b, rtol=1e-10, maxit=20000, precond=precond,
                                              loop=sla.SLA_LOOP_HOST)
        x = torch.full((A.n,), float("nan"), dtype=torch.float64, device=b.device)
        info = _static_solve(dA, b, 1e-10, 20000, precond, x)
        assert info.status == info_ref.status == 0
        assert info.iters == info_ref.iters
        assert rel(x.cpu().numpy(), x_ref.cpu().numpy()) <= X_TOL_F64


def test_static_scratch_rejects_oversized_systems():
    lib = sla.lib()
    A = _abi.sla_csr()
    A.n, A.nnz, A.rowptr_type, A.dtype = 65537, 65537, 0, 1
    A.row_ptr = A.col_idx = A.values = 0x10000
    o = _abi.sla_cg_opts()
    o.rtol, o.maxit = 1e-8, 10
    st = lib.sla_cg_solve_static(ctypes.byref(A), 0x10000, None, ctypes.byref(o), 0x10000, None, None, None)
    assert st == _abi.SLA_WORKSPACE_TOO_SMALL
