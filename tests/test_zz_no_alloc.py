"""The allocation-free solve entry point (sla_cg_solve_static), called through the C ABI.

Some callers cannot allocate device memory: a plugin inside an application that owns and
budgets all device memory, a latency-critical path where an allocation (and the synchronisation
it can imply) is not allowed, a binding with no device allocator.  sla_cg_solve_static serves
them from a fixed scratch array inside the library (at most 65,536 unknowns).  These tests check
that it gives the results of the workspace entry point and of the oracle, that a call changes
the GPU's free memory by nothing, and that it refuses larger systems.

This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import sla, oracle, torch, rel, to_dev, t, check_history, X_TOL_F64, TOL_F32
from differentiable_sparse_iterative_gb300 import _abi
from workloads import diffusion_dirichlet, poisson_5pt

pytestmark = pytest.mark.gpu


def _static_solve(A, b, rtol, maxit, precond, x, x0=None, history=None):
    lib = sla.lib()
    o = _abi.sla_cg_opts()
    o.rtol, o.maxit, o.precond, o.unroll, o.loop, o.reserved = rtol, maxit, precond, 0, 0, 0
    info = _abi.sla_cg_info()
    st = lib.sla_cg_solve_static(ctypes.byref(sla._csr_struct(A)), b.data_ptr(),
                                 None if x0 is None else x0.data_ptr(), ctypes.byref(o), x.data_ptr(),
                                 ctypes.byref(info), None if history is None else history.data_ptr(),
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


def test_static_scratch_exact_fit_fp64_jacobi_against_oracle():
    # n = 65,536 with fp64 values and Jacobi: the layout that fills the scratch array exactly
    m = 256
    A = diffusion_dirichlet(m, np.random.default_rng(7).lognormal(0, 0.5, 2 * m * (m + 1)))
    assert A.n == 65536
    dA = to_dev(A)
    rng = np.random.default_rng(8)
    for _ in range(2):
        bn = rng.standard_normal(A.n)
        x = torch.full((A.n,), float("nan"), dtype=torch.float64, device="cuda:0")
        h = torch.full((20001,), float("nan"), dtype=torch.float64, device="cuda:0")
        info = _static_solve(dA, t(bn), 1e-10, 20000, 1, x, history=h)
        ref = oracle.cg(A.row_ptr, A.col_idx, A.values, bn, rtol=1e-10, maxit=20000, precond=1, history=True)
        assert info.status == ref["status"] == 0
        assert abs(info.iters - ref["iters"]) <= 1
        assert rel(x.cpu().numpy(), ref["x"]) <= X_TOL_F64
        check_history(h.cpu().numpy()[: info.iters + 1], ref["history"], k=50)


def test_static_scratch_fp32_int64_rowptr_x0_history_against_oracle():
    m = 120
    A = poisson_5pt(m, rowptr64=True)
    assert A.row_ptr.dtype == np.int64
    dA = to_dev(A, np.float32)
    rng = np.random.default_rng(9)
    bn = rng.standard_normal(A.n).astype(np.float32)
    x0n = (0.1 * rng.standard_normal(A.n)).astype(np.float32)
    x = torch.zeros(A.n, dtype=torch.float32, device="cuda:0")
    h = torch.full((5001,), float("nan"), dtype=torch.float64, device="cuda:0")
    info = _static_solve(dA, t(bn), 1e-5, 5000, 0, x, x0=t(x0n), history=h)
    ref = oracle.cg(A.row_ptr, A.col_idx, A.values, bn.astype(np.float64), x0=x0n.astype(np.float64), rtol=1e-5,
                    maxit=5000, history=True)
    assert info.status == ref["status"] == 0
    assert abs(info.iters - ref["iters"]) <= max(1, 0.06 * ref["iters"])
    assert rel(x.cpu().numpy(), ref["x"]) <= TOL_F32
    check_history(h.cpu().numpy()[: info.iters + 1], ref["history"], k=10, tol=1e-4)


def test_static_call_allocates_no_device_memory():
    m = 200
    A = poisson_5pt(m)
    dA = to_dev(A)
    b = t(np.random.default_rng(10).standard_normal(A.n))
    x = torch.zeros(A.n, dtype=torch.float64, device="cuda:0")
    _static_solve(dA, b, 1e-10, 20000, 1, x)  # first call: loads the code, looks up the scratch address
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    info = _static_solve(dA, b, 1e-10, 20000, 1, x)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert info.status == 0
    assert free1 == free0, (free0, free1)


def test_static_scratch_rejects_oversized_systems():
    lib = sla.lib()
    A = _abi.sla_csr()
    A.n, A.nnz, A.rowptr_type, A.dtype = 65537, 65537, 0, 1
    A.row_ptr = A.col_idx = A.values = 0x10000
    o = _abi.sla_cg_opts()
    o.rtol, o.maxit = 1e-8, 10
    st = lib.sla_cg_solve_static(ctypes.byref(A), 0x10000, None, ctypes.byref(o), 0x10000, None, None, None)
    assert st == _abi.SLA_WORKSPACE_TOO_SMALL
    # the same argument checks as sla_cg_solve: an int32 row_ptr cannot index 2^31 entries
    A.n, A.nnz = 100, 1 << 31
    st = lib.sla_cg_solve_static(ctypes.byref(A), 0x10000, None, ctypes.byref(o), 0x10000, None, None, None)
    assert st == _abi.SLA_INVALID_ARG
