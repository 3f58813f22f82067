"""libsla loads and exports every symbol include/sla.h declares; host-side argument checks (CPU only)."""
import ctypes
import os
import re

import pytest

from differentiable_sparse_iterative_gb300 import _abi, build as sla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sla_build.build()
    return _abi.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "sla.h")).read()
    return sorted(set(re.findall(r"SLA_API\s+[\w\s\*]*?\b(sla_\w+)\s*\(", text)))


def test_header_matches_binding():
    assert declared_symbols() == sorted(_abi.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and nothing else of ours is visible
    out = os.popen(f"nm -D --defined-only {_abi.LIB_PATH}").read()
    ours = sorted(set(re.findall(r" T (sla_\w+)", out)))
    assert ours == declared_symbols()


def test_status_strings_and_version(lib):
    assert lib.sla_version() == 100
    assert lib.sla_status_string(0) == b"SLA_OK"
    assert lib.sla_status_string(2) == b"SLA_BREAKDOWN"
    assert lib.sla_status_string(99) == b"SLA_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    f = lib.sla_cg_workspace_bytes
    assert f(-1, 1, 1, 0) == 0 and f(10, 0, 1, 0) == 0 and f(10, 1, 7, 0) == 0 and f(10, 1, 1, 5) == 0
    a, j = f(1000, 1, 1, 0), f(1000, 1, 1, 1)
    assert j > a > 4 * 1000 * 8
    assert f(1000, 1, 0, 0) < a                 # float32 vectors are half the size
    assert f(1000, 4, 1, 0) > 3 * (a - 200000)  # batch scales the vectors
    assert a % 256 == 0


def _csr(n=4, nnz=10, rt=0, dt=1, ptr=0x10000):
    A = _abi.sla_csr()
    A.n, A.nnz, A.rowptr_type, A.dtype = n, nnz, rt, dt
    A.row_ptr = A.col_idx = A.values = ptr
    return A


def _opts(rtol=1e-8, maxit=10, precond=0, loop=0, reserved=0, unroll=0):
    o = _abi.sla_cg_opts()
    o.rtol, o.maxit, o.precond, o.unroll, o.loop, o.reserved = rtol, maxit, precond, unroll, loop, reserved
    return o


def _no_gpu_here():
    # these tests hand the library fake device pointers: they must never run where a kernel could
    # actually be launched, so they are skipped on a machine with a GPU
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("fake-pointer ABI checks run only on machines without a GPU")
    except ImportError:
        pass


def test_argument_rejection_without_gpu(lib):
    _no_gpu_here()
    P = 0x10000  # never dereferenced: every case is rejected before any CUDA call
    solve = lib.sla_cg_solve
    assert solve(None, P, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == _abi.SLA_INVALID_ARG
    assert solve(ctypes.byref(_csr(dt=7)), P, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr(rt=9)), P, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr(n=-1)), P, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr(n=1 << 31)), P, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), P, None, None, P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(rtol=-1.0)), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(rtol=float("nan"))), P, None, None, P,
                 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(maxit=-1)), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(precond=3)), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(loop=4)), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(reserved=1)), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts(unroll=65)), P, None, None, P, 1 << 20,
                 None) == 3
    assert solve(ctypes.byref(_csr()), None, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P + 4, None, ctypes.byref(_opts()), P, None, None, P, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts()), P, None, None, P + 16, 1 << 20, None) == 3
    assert solve(ctypes.byref(_csr()), P, None, ctypes.byref(_opts()), P, None, None, P, 16,
                 None) == _abi.SLA_WORKSPACE_TOO_SMALL
    assert lib.sla_cg_solve_batched(ctypes.byref(_csr()), -1, P, P, None, ctypes.byref(_opts()), P, None, None,
                                    P, 1 << 20, None) == 3
    assert lib.sla_spmv(ctypes.byref(_csr(rt=0, nnz=1 << 31)), P, P, None) == 3


def test_empty_system_needs_no_gpu(lib):
    _no_gpu_here()
    info = _abi.sla_cg_info()
    info.status = 77
    st = lib.sla_cg_solve(ctypes.byref(_csr(n=0, nnz=0)), None, None, ctypes.byref(_opts()), None,
                          ctypes.byref(info), None, None, 0, None)
    assert st == 0 and info.status == 0 and info.iters == 0
    assert lib.sla_cg_solve_batched(ctypes.byref(_csr()), 0, 0x10000, 0x10000, None, ctypes.byref(_opts()),
                                    0x10000, None, None, 0x10000, 1 << 20, None) == 0


def _eig_opts(tol=1e-10, maxit=10, inner_factor=0.01, inner_maxit=100, precond=0, loop=0):
    o = _abi.sla_eig_opts()
    o.tol, o.maxit, o.inner_factor, o.inner_maxit, o.precond, o.loop = tol, maxit, inner_factor, inner_maxit, \
        precond, loop
    return o


def test_eig_workspace_bytes(lib):
    f = lib.sla_eig_workspace_bytes
    assert f(-1, 1, 0) == 0 and f(10, 7, 0) == 0 and f(10, 1, 5) == 0
    n = 1000
    assert f(n, 1, 0) >= lib.sla_cg_workspace_bytes(n, 1, 1, 0) + 2 * 8 * n
    assert f(n, 1, 1) > f(n, 1, 0) > f(n, 0, 0)
    assert f(n, 1, 0) % 256 == 0


def test_eig_argument_rejection_without_gpu(lib):
    _no_gpu_here()
    P = 0x10000  # never dereferenced: every case is rejected before any CUDA call
    ws = 1 << 24
    info = _abi.sla_eig_info()
    eig = lib.sla_eig_smallest
    ok = ctypes.byref(_eig_opts())
    assert eig(None, P, ok, ctypes.byref(info), P, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), P, None, ctypes.byref(info), P, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), P, ok, None, P, ws, None) == _abi.SLA_INVALID_ARG
    for bad in [dict(tol=-1.0), dict(tol=float("nan")), dict(maxit=-1), dict(inner_factor=0.0),
                dict(inner_factor=1.0), dict(inner_maxit=-1), dict(precond=2), dict(loop=9)]:
        assert eig(ctypes.byref(_csr()), P, ctypes.byref(_eig_opts(**bad)), ctypes.byref(info), P, ws,
                   None) == _abi.SLA_INVALID_ARG, bad
    assert eig(ctypes.byref(_csr(n=0, nnz=0)), P, ok, ctypes.byref(info), P, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), None, ok, ctypes.byref(info), P, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), P + 4, ok, ctypes.byref(info), P, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), P, ok, ctypes.byref(info), P + 16, ws, None) == _abi.SLA_INVALID_ARG
    assert eig(ctypes.byref(_csr()), P, ok, ctypes.byref(info), P, 64, None) == _abi.SLA_WORKSPACE_TOO_SMALL
    grad = lib.sla_eig_grad_values
    assert grad(ctypes.byref(_csr()), -1, P, None, P, None) == _abi.SLA_INVALID_ARG
    assert grad(ctypes.byref(_csr()), 17, P, None, P, None) == _abi.SLA_INVALID_ARG
    assert grad(ctypes.byref(_csr()), 1, None, None, P, None) == _abi.SLA_INVALID_ARG
    assert grad(ctypes.byref(_csr()), 1, P, None, None, None) == _abi.SLA_INVALID_ARG
    assert grad(ctypes.byref(_csr(nnz=0)), 1, P, None, None, None) == _abi.SLA_OK  # nothing to write


def test_tuning_and_test_hooks_reject_bad_values(lib):
    # process-wide switches: no GPU needed to refuse an unknown value
    e, b_, u = (ctypes.c_int64(-1) for _ in range(3))  # no CUDA call: counters of this process
    assert lib.sla_graph_cache_stats(ctypes.byref(e), ctypes.byref(b_), ctypes.byref(u)) == _abi.SLA_OK
    assert 0 <= e.value <= 32 and e.value <= b_.value and u.value >= 0
    assert lib.sla_graph_cache_stats(None, None, None) == _abi.SLA_OK
    assert lib.sla_set_spmv_variant(2) == _abi.SLA_INVALID_ARG
    assert lib.sla_set_spmv_variant(-1) == _abi.SLA_INVALID_ARG
    assert lib.sla_set_spmv_variant(_abi.SLA_SPMV_PLAIN) == _abi.SLA_OK
    assert lib.sla_test_set_barrier_wait(2, 0) == _abi.SLA_INVALID_ARG
    assert lib.sla_test_set_barrier_wait(0, -5) == _abi.SLA_INVALID_ARG
    assert lib.sla_test_set_barrier_wait(0, (1 << 26) + 1) == _abi.SLA_INVALID_ARG
    assert lib.sla_test_set_barrier_wait(0, 0) == _abi.SLA_OK


def test_library_reads_no_environment_variables():
    # the solver's behaviour is set through the C ABI only: no getenv in the library sources
    csrc = os.path.join(ROOT, "differentiable_sparse_iterative_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "getenv" not in open(os.path.join(csrc, f)).read(), f


def test_bicgstab_workspace_bytes(lib):
    f = lib.sla_bicgstab_workspace_bytes
    assert f(-1, 0, 1) == 0 and f(10, -1, 1) == 0 and f(10, 10, 7) == 0
    n, nnz = 100_000, 500_000
    f64, f32 = f(n, nnz, 1), f(n, nnz, 0)
    # eight n-vectors, the transposed values, A^T's column indices, row pointers and column counts
    assert f64 >= 8 * 8 * n + 8 * nnz + 4 * nnz + 8 * (n + 1) + 4 * n
    assert f32 >= 8 * 4 * n + 4 * nnz + 4 * nnz + 8 * (n + 1) + 4 * n
    assert f64 > f32 and f(n, 2 * nnz, 1) - f64 >= (8 + 4) * nnz - 512
    assert f(0, 0, 1) > 0  # the control block and the reductions' scratch
