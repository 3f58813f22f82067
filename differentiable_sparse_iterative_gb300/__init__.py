"""Differentiable sparse iterative solve on GB300: Python binding of libsla.

The compute runs in libsla's CUDA kernels (``csrc/``, C ABI in ``include/sla.h``);
this module only marshals torch tensors (device memory, the current stream) into
the C calls, under the same names.  There is no CPU or PyTorch fallback: if
libsla.so is missing or a tensor is not on a CUDA device the call raises.

Method: "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers and
Sparse Tensor Parallelism for PyTorch" (Chi, Wen), technical summary —
Methodology 1 (autograd-aware .matvec / .solve; one matrix or a batch sharing a
pattern), Methodology 2 (adjoint: one A^T lambda = dL/dx solve, grad_b = lambda,
grad_A = -lambda_i x_j on the pattern, O(1) graph nodes; eigenvalue problems:
d mu / d A_ij = v_i v_j on the pattern), Significance (Jacobi preconditioning).

    A = CSRMatrix(row_ptr, col_idx, values)          # CUDA tensors
    x = solve(A, b, rtol=1e-8)                       # autograd: grads to values and b
"""
from __future__ import annotations

import ctypes
import warnings
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import _abi
from ._abi import (SLA_OK, SLA_NOT_CONVERGED, SLA_BREAKDOWN, SLA_INVALID_ARG, SLA_BAD_CSR, SLA_NONFINITE,
                   SLA_WORKSPACE_TOO_SMALL, SLA_TIMEOUT, SLA_CUDA_ERROR, SLA_PRECOND_NONE, SLA_PRECOND_JACOBI, SLA_LOOP_AUTO,
                   SLA_LOOP_HOST, SLA_LOOP_GRAPH, SLA_LOOP_RESIDENT, SLA_LOOP_CLUSTER)

__all__ = [
    "CSRMatrix", "SlaError", "CGInfo", "lib", "sla_spmv", "sla_cg_solve", "sla_cg_adjoint", "sla_grad_values",
    "sla_cg_solve_batched", "sla_cg_adjoint_batched", "sla_validate_csr", "sla_cg_workspace_bytes",
    "sla_status_string", "sla_launch_count", "sla_version", "CGSolve", "solve", "CGSolveBatched", "solve_batched", "sla_bicgstab_workspace_bytes", "sla_bicgstab_solve",
    "sla_bicgstab_adjoint", "BiCGStabSolve", "sla_eigsh", "sla_eigsh_workspace_bytes", "Eigsh", "eigsh",
    "matvec",
    "SLA_PRECOND_NONE", "SLA_PRECOND_JACOBI", "SLA_LOOP_AUTO", "SLA_LOOP_HOST", "SLA_LOOP_GRAPH",
    "SLA_LOOP_RESIDENT", "SLA_LOOP_CLUSTER", "SLA_OK", "SLA_NOT_CONVERGED", "SLA_BREAKDOWN", "SLA_INVALID_ARG",
    "SLA_BAD_CSR", "SLA_NONFINITE", "SLA_WORKSPACE_TOO_SMALL", "SLA_TIMEOUT", "SLA_CUDA_ERROR",
    "EigInfo", "sla_eig_workspace_bytes", "sla_eig_smallest", "sla_eig_grad_values", "EigSmallest",
    "eigsh_smallest", "sla_spmv_transpose", "sla_matvec_grad_values", "MatVec", "sla_set_spmv_variant", "sla_graph_cache_stats", "sla_test_set_barrier_wait", "SLA_SPMV_PLAIN", "SLA_SPMV_TMA",
]
from ._abi import SLA_SPMV_PLAIN, SLA_SPMV_TMA  # noqa: E402

_lib = None


def lib():
    """The loaded libsla (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = _abi.load()
    return _lib


class SlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {sla_status_string(status)}"
        if status == SLA_CUDA_ERROR:
            msg += f" ({lib().sla_last_cuda_error().decode()})"
        super().__init__(msg)
        self.status = status


PATHS = {1: "host", 2: "graph", 3: "resident", 4: "cluster"}


@dataclass
class CGInfo:
    iters: int
    rel_res: float
    status: int
    kernels: int
    path: str = ""

    @property
    def status_name(self) -> str:
        return sla_status_string(self.status)


@dataclass
class CSRMatrix:
    """Square CSR matrix on a CUDA device: row_ptr (int32/int64, n+1), col_idx (int32), values (f32/f64)."""
    row_ptr: torch.Tensor
    col_idx: torch.Tensor
    values: torch.Tensor

    @property
    def n(self) -> int:
        return self.row_ptr.shape[0] - 1

    @property
    def nnz(self) -> int:
        return self.col_idx.shape[0]

    @classmethod
    def from_numpy(cls, row_ptr, col_idx, values, device="cuda"):
        return cls(torch.as_tensor(row_ptr).to(device), torch.as_tensor(col_idx).to(device),
                   torch.as_tensor(values).to(device))

    def with_values(self, values: torch.Tensor) -> "CSRMatrix":
        return CSRMatrix(self.row_ptr, self.col_idx, values)

    # The method-style interface of the pages' sparse tensor (A.solve(f), A.matvec(x), A.eigsh()),
    # each the differentiable module function of the same name.
    def solve(self, b: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000, precond: int = 0,
              method: str = "cg") -> torch.Tensor:
        """Differentiable x = A^{-1} b (see solve)."""
        return solve(self, b, rtol=rtol, maxit=maxit, precond=precond, method=method)

    def matvec(self, x: torch.Tensor) -> torch.Tensor:
        """Differentiable y = A x (see matvec)."""
        return matvec(self, x)

    def eigsh(self, k: Optional[int] = None, **kw):
        """Without k: the smallest eigenpair (mu, v) (see eigsh_smallest).  With k: the k smallest
        (mu [k], V [k, n]) (see eigsh).  mu is differentiable with respect to the values; the
        keyword arguments are those of the function called."""
        return eigsh_smallest(self, **kw) if k is None else eigsh(self, k, **kw)


_DT = {torch.float32: _abi.SLA_F32, torch.float64: _abi.SLA_F64}
_IT = {torch.int32: _abi.SLA_I32, torch.int64: _abi.SLA_I64}


def _dev_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libsla has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


def _csr_struct(A: CSRMatrix, values: Optional[torch.Tensor] = None) -> _abi.sla_csr:
    vals = A.values if values is None else values
    if vals.dtype not in _DT:
        raise ValueError("values must be float32 or float64")
    if A.row_ptr.dtype not in _IT or A.col_idx.dtype != torch.int32:
        raise ValueError("row_ptr must be int32/int64 and col_idx int32")
    s = _abi.sla_csr()
    s.n = A.n
    s.nnz = A.nnz
    s.rowptr_type = _IT[A.row_ptr.dtype]
    s.dtype = _DT[vals.dtype]
    s.row_ptr = _dev_ptr(A.row_ptr, name="row_ptr")
    s.col_idx = _dev_ptr(A.col_idx, name="col_idx")
    s.values = _dev_ptr(vals, name="values") if vals.dim() == 1 else None
    return s


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _opts(rtol, maxit, precond, unroll=0, loop=SLA_LOOP_AUTO) -> _abi.sla_cg_opts:
    o = _abi.sla_cg_opts()
    o.rtol = float(rtol)
    o.maxit = int(maxit)
    o.precond = int(precond)
    o.unroll = int(unroll)
    o.loop = int(loop)
    o.reserved = 0
    return o


def _check(st: int, where: str):
    if st != SLA_OK:
        raise SlaError(st, where)


def sla_status_string(status: int) -> str:
    return lib().sla_status_string(int(status)).decode()


def sla_version() -> int:
    return lib().sla_version()


def sla_set_spmv_variant(variant: int) -> None:
    """Process-wide SpMV step of the GRAPH and HOST loops: SLA_SPMV_PLAIN (default) or SLA_SPMV_TMA."""
    _check(lib().sla_set_spmv_variant(int(variant)), "sla_set_spmv_variant")


def sla_graph_cache_stats() -> Tuple[int, int, int]:
    """(cached graph loops, graphs instantiated, in-place argument replacements) of this process."""
    e, b, u = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().sla_graph_cache_stats(ctypes.byref(e), ctypes.byref(b), ctypes.byref(u)), "sla_graph_cache_stats")
    return int(e.value), int(b.value), int(u.value)


def sla_test_set_barrier_wait(extra: int, spin_limit: int) -> None:
    """Test hook: the resident grid barrier waits for `extra` more arrivals, at most `spin_limit` polls."""
    _check(lib().sla_test_set_barrier_wait(int(extra), int(spin_limit)), "sla_test_set_barrier_wait")


def sla_launch_count() -> int:
    return lib().sla_launch_count()


def sla_cg_workspace_bytes(n: int, batch: int, dtype: torch.dtype, precond: int) -> int:
    return lib().sla_cg_workspace_bytes(int(n), int(batch), _DT[dtype], int(precond))


def _workspace(n, batch, dtype, precond, device, ws: Optional[torch.Tensor]) -> torch.Tensor:
    need = sla_cg_workspace_bytes(n, batch, dtype, precond)
    if ws is not None and ws.numel() * ws.element_size() >= need:
        return ws
    return torch.empty(max(need, 256), dtype=torch.uint8, device=device)


def sla_validate_csr(A: CSRMatrix, check_symmetric: bool = False) -> int:
    """Returns -1 when A is canonical (and symmetric if asked), else the first offending row."""
    ws = torch.empty(256, dtype=torch.uint8, device=A.row_ptr.device)
    bad = ctypes.c_int64(-1)
    st = lib().sla_validate_csr(ctypes.byref(_csr_struct(A)), int(bool(check_symmetric)), ctypes.byref(bad),
                                ws.data_ptr(), 256, _stream(A.row_ptr.device))
    if st not in (SLA_OK, SLA_BAD_CSR):
        _check(st, "sla_validate_csr")
    return int(bad.value)


def sla_spmv(A: CSRMatrix, x: torch.Tensor, y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y = A x (asynchronous on the current stream)."""
    if y is None:
        y = torch.empty(A.n, dtype=A.values.dtype, device=A.values.device)
    _check(lib().sla_spmv(ctypes.byref(_csr_struct(A)), _dev_ptr(x, A.values.dtype, "x"),
                          _dev_ptr(y, A.values.dtype, "y"), _stream(A.values.device)), "sla_spmv")
    return y


def sla_grad_values(A: CSRMatrix, lam: torch.Tensor, x: torch.Tensor,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad_values[k] = -lam[row(k)] * x[col(k)] on A's pattern (asynchronous)."""
    if out is None:
        out = torch.empty(A.nnz, dtype=A.values.dtype, device=A.values.device)
    _check(lib().sla_grad_values(ctypes.byref(_csr_struct(A)), _dev_ptr(lam, A.values.dtype, "lambda"),
                                 _dev_ptr(x, A.values.dtype, "x"), _dev_ptr(out, A.values.dtype, "grad_values"),
                                 _stream(A.values.device)), "sla_grad_values")
    return out


def _info(ci: _abi.sla_cg_info) -> CGInfo:
    return CGInfo(int(ci.iters), float(ci.rel_res), int(ci.status), int(ci.kernels), PATHS.get(int(ci.path), ""))


def sla_cg_solve(A: CSRMatrix, b: torch.Tensor, x0: Optional[torch.Tensor] = None, rtol: float = 1e-8,
                 maxit: int = 10000, precond: int = SLA_PRECOND_NONE, x: Optional[torch.Tensor] = None,
                 history: bool = False, workspace: Optional[torch.Tensor] = None, sync: bool = True,
                 unroll: int = 0, loop: int = SLA_LOOP_AUTO):
    """CG solve of A x = b.  Returns (x, CGInfo or None, history tensor or None).

    With sync=False the call is asynchronous and returns info=None.
    """
    dt, dev = A.values.dtype, A.values.device
    if x is None:
        x = torch.empty(A.n, dtype=dt, device=dev)
    hist = torch.full((int(maxit) + 1,), float("nan"), dtype=torch.float64, device=dev) if history else None
    ws = _workspace(A.n, 1, dt, precond, dev, workspace)
    info = _abi.sla_cg_info()
    st = lib().sla_cg_solve(ctypes.byref(_csr_struct(A)), _dev_ptr(b, dt, "b"), _dev_ptr(x0, dt, "x0"),
                            ctypes.byref(_opts(rtol, maxit, precond, unroll, loop)), _dev_ptr(x, dt, "x"),
                            ctypes.byref(info) if sync else None, _dev_ptr(hist, torch.float64, "history"),
                            ws.data_ptr(), ws.numel(), _stream(dev))
    _check(st, "sla_cg_solve")
    return x, (_info(info) if sync else None), hist


def sla_cg_adjoint(A: CSRMatrix, x: torch.Tensor, g: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000,
                   precond: int = SLA_PRECOND_NONE, grad_b: Optional[torch.Tensor] = None,
                   grad_values: Optional[torch.Tensor] = None, want_grad_values: bool = True,
                   workspace: Optional[torch.Tensor] = None, sync: bool = True, unroll: int = 0,
                   loop: int = SLA_LOOP_AUTO):
    """Adjoint backward: returns (grad_b = lambda, grad_values or None, CGInfo or None)."""
    dt, dev = A.values.dtype, A.values.device
    if grad_b is None:
        grad_b = torch.empty(A.n, dtype=dt, device=dev)
    if grad_values is None and want_grad_values:
        grad_values = torch.empty(A.nnz, dtype=dt, device=dev)
    ws = _workspace(A.n, 1, dt, precond, dev, workspace)
    info = _abi.sla_cg_info()
    st = lib().sla_cg_adjoint(ctypes.byref(_csr_struct(A)), _dev_ptr(x, dt, "x"), _dev_ptr(g, dt, "g"),
                              ctypes.byref(_opts(rtol, maxit, precond, unroll, loop)), _dev_ptr(grad_b, dt, "grad_b"),
                              _dev_ptr(grad_values, dt, "grad_values"), ctypes.byref(info) if sync else None,
                              ws.data_ptr(), ws.numel(), _stream(dev))
    _check(st, "sla_cg_adjoint")
    return grad_b, grad_values, (_info(info) if sync else None)


def sla_cg_solve_batched(pattern: CSRMatrix, values: torch.Tensor, b: torch.Tensor,
                         x0: Optional[torch.Tensor] = None, rtol: float = 1e-5, maxit: int = 10000,
                         precond: int = SLA_PRECOND_NONE, x: Optional[torch.Tensor] = None, history: bool = False,
                         workspace: Optional[torch.Tensor] = None, sync: bool = True, unroll: int = 0,
                         loop: int = SLA_LOOP_AUTO):
    """Batched shared-pattern CG: values [B, nnz], b [B, n].  Returns (x [B, n], [CGInfo]*B, history)."""
    B = values.shape[0]
    dt, dev = values.dtype, values.device
    if x is None:
        x = torch.empty(B, pattern.n, dtype=dt, device=dev)
    hist = (torch.full((B, int(maxit) + 1), float("nan"), dtype=torch.float64, device=dev) if history else None)
    ws = _workspace(pattern.n, B, dt, precond, dev, workspace)
    infos = (_abi.sla_cg_info * max(B, 1))()
    st = lib().sla_cg_solve_batched(ctypes.byref(_csr_struct(pattern, values)), B, _dev_ptr(values, dt, "values"),
                                    _dev_ptr(b, dt, "b"), _dev_ptr(x0, dt, "x0"),
                                    ctypes.byref(_opts(rtol, maxit, precond, unroll, loop)), _dev_ptr(x, dt, "x"),
                                    infos if sync else None, _dev_ptr(hist, torch.float64, "history"),
                                    ws.data_ptr(), ws.numel(), _stream(dev))
    _check(st, "sla_cg_solve_batched")
    return x, ([_info(infos[s]) for s in range(B)] if sync else None), hist


def sla_cg_adjoint_batched(pattern: CSRMatrix, values: torch.Tensor, x: torch.Tensor, g: torch.Tensor,
                           rtol: float = 1e-5, maxit: int = 10000, precond: int = SLA_PRECOND_NONE,
                           grad_b: Optional[torch.Tensor] = None, grad_values: Optional[torch.Tensor] = None,
                           want_grad_values: bool = True, workspace: Optional[torch.Tensor] = None,
                           sync: bool = True, unroll: int = 0, loop: int = SLA_LOOP_AUTO):
    """Batched adjoint: returns (grad_b [B, n], grad_values [B, nnz] or None, [CGInfo]*B)."""
    B = values.shape[0]
    dt, dev = values.dtype, values.device
    if grad_b is None:
        grad_b = torch.empty(B, pattern.n, dtype=dt, device=dev)
    if grad_values is None and want_grad_values:
        grad_values = torch.empty(B, pattern.nnz, dtype=dt, device=dev)
    ws = _workspace(pattern.n, B, dt, precond, dev, workspace)
    infos = (_abi.sla_cg_info * max(B, 1))()
    st = lib().sla_cg_adjoint_batched(ctypes.byref(_csr_struct(pattern, values)), B, _dev_ptr(values, dt, "values"),
                                      _dev_ptr(x, dt, "x"), _dev_ptr(g, dt, "g"),
                                      ctypes.byref(_opts(rtol, maxit, precond, unroll, loop)),
                                      _dev_ptr(grad_b, dt, "grad_b"), _dev_ptr(grad_values, dt, "grad_values"),
                                      infos if sync else None, ws.data_ptr(), ws.numel(), _stream(dev))
    _check(st, "sla_cg_adjoint_batched")
    return grad_b, grad_values, ([_info(infos[s]) for s in range(B)] if sync else None)


def _raise_on_failure(info: CGInfo, where: str):
    if info.status == SLA_NOT_CONVERGED:
        warnings.warn(f"{where}: CG did not reach rtol in {info.iters} iterations (rel_res {info.rel_res:.3e})")
    elif info.status != SLA_OK:
        raise SlaError(info.status, where)


class CGSolve(torch.autograd.Function):
    """x = A^{-1} b with the adjoint backward (one node in the autograd graph).

    Saved for backward: x and A (pattern and values): O(n + nnz), whatever the
    iteration count.  Backward solves A lambda = dL/dx with the same rtol, maxit
    and preconditioner and returns grad_values = -lambda_i x_j on the pattern and
    grad_b = lambda.
    """

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, b, rtol, maxit, precond):
        A = CSRMatrix(row_ptr, col_idx, values)
        x, info, _ = sla_cg_solve(A, b, rtol=rtol, maxit=maxit, precond=precond)
        _raise_on_failure(info, "CGSolve.forward")
        ctx.save_for_backward(row_ptr, col_idx, values, x)
        ctx.opts = (rtol, maxit, precond)
        ctx.fwd_info = info
        return x

    @staticmethod
    def backward(ctx, g):
        row_ptr, col_idx, values, x = ctx.saved_tensors
        rtol, maxit, precond = ctx.opts
        A = CSRMatrix(row_ptr, col_idx, values)
        need_v, need_b = ctx.needs_input_grad[2], ctx.needs_input_grad[3]
        grad_b, grad_v, info = sla_cg_adjoint(A, x, g.contiguous(), rtol=rtol, maxit=maxit, precond=precond,
                                              want_grad_values=need_v)
        _raise_on_failure(info, "CGSolve.backward")
        return None, None, (grad_v if need_v else None), (grad_b if need_b else None), None, None, None


def sla_bicgstab_workspace_bytes(n: int, nnz: int, dtype: torch.dtype) -> int:
    return lib().sla_bicgstab_workspace_bytes(int(n), int(nnz), _DT[dtype])


def _bi_workspace(A: CSRMatrix, ws: Optional[torch.Tensor]) -> torch.Tensor:
    need = sla_bicgstab_workspace_bytes(A.n, A.nnz, A.values.dtype)
    if ws is not None and ws.numel() * ws.element_size() >= need:
        return ws
    return torch.empty(max(need, 256), dtype=torch.uint8, device=A.values.device)


def sla_bicgstab_solve(A: CSRMatrix, b: torch.Tensor, x0: Optional[torch.Tensor] = None, rtol: float = 1e-8,
                       maxit: int = 10000, x: Optional[torch.Tensor] = None, history: bool = False,
                       workspace: Optional[torch.Tensor] = None, unroll: int = 0, loop: int = SLA_LOOP_AUTO):
    """BiCGStab solve of a general A x = b.  Returns (x, CGInfo, history tensor or None).  loop:
    SLA_LOOP_HOST runs the host-driven kernel loop, any other value the resident kernel (the host
    loop when it cannot be launched)."""
    dt, dev = A.values.dtype, A.values.device
    if x is None:
        x = torch.empty(A.n, dtype=dt, device=dev)
    hist = torch.full((int(maxit) + 1,), float("nan"), dtype=torch.float64, device=dev) if history else None
    ws = _bi_workspace(A, workspace)
    info = _abi.sla_cg_info()
    st = lib().sla_bicgstab_solve(ctypes.byref(_csr_struct(A)), _dev_ptr(b, dt, "b"), _dev_ptr(x0, dt, "x0"),
                                  ctypes.byref(_opts(rtol, maxit, SLA_PRECOND_NONE, unroll, loop)), _dev_ptr(x, dt, "x"),
                                  ctypes.byref(info), _dev_ptr(hist, torch.float64, "history"), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream(dev))
    _check(st, "sla_bicgstab_solve")
    return x, _info(info), hist


def sla_bicgstab_adjoint(A: CSRMatrix, x: torch.Tensor, g: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000,
                         want_grad_values: bool = True, workspace: Optional[torch.Tensor] = None, unroll: int = 0,
                         loop: int = SLA_LOOP_AUTO):
    """Adjoint of the BiCGStab solve: A^T lambda = g; returns (grad_b = lambda, grad_values or None, CGInfo).
    A^T shares A's pattern when that is structurally symmetric, and is built explicitly otherwise."""
    dt, dev = A.values.dtype, A.values.device
    grad_b = torch.empty(A.n, dtype=dt, device=dev)
    grad_values = torch.empty(A.nnz, dtype=dt, device=dev) if want_grad_values else None
    ws = _bi_workspace(A, workspace)
    info = _abi.sla_cg_info()
    st = lib().sla_bicgstab_adjoint(ctypes.byref(_csr_struct(A)), _dev_ptr(x, dt, "x"), _dev_ptr(g, dt, "g"),
                                    ctypes.byref(_opts(rtol, maxit, SLA_PRECOND_NONE, unroll, loop)),
                                    _dev_ptr(grad_b, dt, "grad_b"), _dev_ptr(grad_values, dt, "grad_values"),
                                    ctypes.byref(info), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(dev))
    _check(st, "sla_bicgstab_adjoint")
    return grad_b, grad_values, _info(info)


class BiCGStabSolve(torch.autograd.Function):
    """x = A^{-1} b for a general A by BiCGStab, with the adjoint backward A^T lambda = dL/dx by the
    same solver: grad_values = -lambda_i x_j on the pattern, grad_b = lambda."""

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, b, rtol, maxit):
        A = CSRMatrix(row_ptr, col_idx, values)
        x, info, _ = sla_bicgstab_solve(A, b.contiguous(), rtol=rtol, maxit=maxit)
        _raise_on_failure(info, "BiCGStabSolve.forward")
        ctx.save_for_backward(row_ptr, col_idx, values, x)
        ctx.opts = (rtol, maxit)
        return x

    @staticmethod
    def backward(ctx, g):
        row_ptr, col_idx, values, x = ctx.saved_tensors
        rtol, maxit = ctx.opts
        A = CSRMatrix(row_ptr, col_idx, values)
        need_v, need_b = ctx.needs_input_grad[2], ctx.needs_input_grad[3]
        grad_b, grad_v, info = sla_bicgstab_adjoint(A, x, g.contiguous(), rtol=rtol, maxit=maxit,
                                                    want_grad_values=need_v)
        _raise_on_failure(info, "BiCGStabSolve.backward")
        return None, None, (grad_v if need_v else None), (grad_b if need_b else None), None, None


def solve(A: CSRMatrix, b: torch.Tensor, rtol: float = 1e-8, maxit: int = 10000,
          precond: int = SLA_PRECOND_NONE, method: str = "cg") -> torch.Tensor:
    """Differentiable x = A^{-1} b (gradients flow to A.values and b).  method "cg": symmetric
    positive definite A (optionally Jacobi preconditioned); "bicgstab": general A, unpreconditioned
    (its backward solves A^T lambda = dL/dx by the same method)."""
    if method == "cg":
        return CGSolve.apply(A.row_ptr, A.col_idx, A.values, b, rtol, maxit, precond)
    if method == "bicgstab":
        if precond != SLA_PRECOND_NONE:
            raise ValueError("bicgstab takes no preconditioner")
        return BiCGStabSolve.apply(A.row_ptr, A.col_idx, A.values, b, rtol, maxit)
    raise ValueError(f"unknown method {method!r} (cg or bicgstab)")


class CGSolveBatched(torch.autograd.Function):
    """X[s] = A_s^{-1} B[s] for a batch of systems sharing one pattern (values [S, nnz], B [S, n]),
    with the batched adjoint backward: grad_values[s] = -lambda_s[i] x_s[j] on the pattern and
    grad_B[s] = lambda_s, lambda_s solving A_s lambda_s = dL/dX[s] with the same rtol, maxit and
    preconditioner.  Saved for backward: the pattern, the values and X (O(S (n + nnz)))."""

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, b, rtol, maxit, precond):
        P = CSRMatrix(row_ptr, col_idx, values[0])
        x, infos, _ = sla_cg_solve_batched(P, values.contiguous(), b.contiguous(), rtol=rtol, maxit=maxit,
                                           precond=precond)
        for s, info in enumerate(infos):
            _raise_on_failure(info, f"CGSolveBatched.forward (system {s})")
        ctx.save_for_backward(row_ptr, col_idx, values, x)
        ctx.opts = (rtol, maxit, precond)
        return x

    @staticmethod
    def backward(ctx, g):
        row_ptr, col_idx, values, x = ctx.saved_tensors
        rtol, maxit, precond = ctx.opts
        P = CSRMatrix(row_ptr, col_idx, values[0])
        need_v, need_b = ctx.needs_input_grad[2], ctx.needs_input_grad[3]
        grad_b, grad_v, infos = sla_cg_adjoint_batched(P, values.contiguous(), x, g.contiguous(), rtol=rtol,
                                                       maxit=maxit, precond=precond, want_grad_values=need_v)
        for s, info in enumerate(infos):
            _raise_on_failure(info, f"CGSolveBatched.backward (system {s})")
        return None, None, (grad_v if need_v else None), (grad_b if need_b else None), None, None, None


def solve_batched(row_ptr: torch.Tensor, col_idx: torch.Tensor, values: torch.Tensor, b: torch.Tensor,
                  rtol: float = 1e-5, maxit: int = 10000, precond: int = SLA_PRECOND_NONE) -> torch.Tensor:
    """Differentiable batched solve over one shared pattern: values [S, nnz], b [S, n] -> x [S, n]
    (gradients flow to values and b)."""
    return CGSolveBatched.apply(row_ptr, col_idx, values, b, rtol, maxit, precond)


def sla_spmv_transpose(A: CSRMatrix, x: torch.Tensor, y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y = A^T x for a structurally symmetric pattern (values may differ); raises SlaError(SLA_BAD_CSR)
    when a stored entry has no stored partner (synchronises the stream to check)."""
    dt, dev = A.values.dtype, A.values.device
    if y is None:
        y = torch.empty(A.n, dtype=dt, device=dev)
    bad = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().sla_spmv_transpose(ctypes.byref(_csr_struct(A)), _dev_ptr(x, dt, "x"), _dev_ptr(y, dt, "y"),
                                    _dev_ptr(bad, name="bad"), _stream(dev)), "sla_spmv_transpose")
    if int(bad.item()) != 0:
        raise SlaError(SLA_BAD_CSR, "sla_spmv_transpose (the pattern is not structurally symmetric)")
    return y


def sla_matvec_grad_values(A: CSRMatrix, gy: torch.Tensor, x: torch.Tensor,
                           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad_values[k] = gy[row(k)] * x[col(k)]: the gradient of L(A x) w.r.t. the stored values (asynchronous)."""
    dt, dev = A.values.dtype, A.values.device
    if out is None:
        out = torch.empty(A.nnz, dtype=dt, device=dev)
    _check(lib().sla_matvec_grad_values(ctypes.byref(_csr_struct(A)), _dev_ptr(gy, dt, "gy"), _dev_ptr(x, dt, "x"),
                                        _dev_ptr(out, dt, "grad_values"), _stream(dev)), "sla_matvec_grad_values")
    return out


class MatVec(torch.autograd.Function):
    """y = A x with gradients to the stored values (gy_i x_j on the pattern) and to x (A^T gy)."""

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, x):
        A = CSRMatrix(row_ptr, col_idx, values)
        y = sla_spmv(A, x.contiguous())
        ctx.save_for_backward(row_ptr, col_idx, values, x)
        return y

    @staticmethod
    def backward(ctx, gy):
        row_ptr, col_idx, values, x = ctx.saved_tensors
        A = CSRMatrix(row_ptr, col_idx, values)
        gy = gy.contiguous()
        gv = sla_matvec_grad_values(A, gy, x.contiguous()) if ctx.needs_input_grad[2] else None
        gx = sla_spmv_transpose(A, gy) if ctx.needs_input_grad[3] else None
        return None, None, gv, gx


def matvec(A: CSRMatrix, x: torch.Tensor) -> torch.Tensor:
    """Differentiable y = A x (gradients flow to A.values and x; the x gradient A^T dL/dy needs a
    structurally symmetric pattern)."""
    return MatVec.apply(A.row_ptr, A.col_idx, A.values, x)


# --------------------------------------------------------------------------- eigenvalue problems

@dataclass
class EigInfo:
    iters: int          # outer steps (inner CG solves)
    inner_iters: int    # CG iterations over all steps
    mu: float
    residual: float     # ||A v - mu v||
    status: int

    @property
    def status_name(self) -> str:
        return sla_status_string(self.status)


def sla_eig_workspace_bytes(n: int, dtype: torch.dtype, precond: int = SLA_PRECOND_NONE) -> int:
    return lib().sla_eig_workspace_bytes(int(n), _DT[dtype], int(precond))


def sla_eig_smallest(A: CSRMatrix, v0: Optional[torch.Tensor] = None, tol: Optional[float] = None,
                     maxit: int = 1000, inner_factor: float = 0.01, inner_maxit: int = 100000,
                     precond: int = SLA_PRECOND_NONE, loop: int = SLA_LOOP_AUTO,
                     workspace: Optional[torch.Tensor] = None):
    """Smallest eigenpair of SPD A by inverse iteration on the CG.  Returns (mu, v, EigInfo).

    v0 defaults to all ones (for a diffusion or Laplace operator it overlaps the positive
    fundamental mode); tol defaults to 1e-10 for float64 and 1e-5 for float32 data.
    """
    dt, dev = A.values.dtype, A.values.device
    if tol is None:
        tol = 1e-10 if dt == torch.float64 else 1e-5
    v = torch.ones(A.n, dtype=dt, device=dev) if v0 is None else v0.detach().clone()
    need = sla_eig_workspace_bytes(A.n, dt, precond)
    ws = workspace if workspace is not None and workspace.numel() * workspace.element_size() >= need else \
        torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    o = _abi.sla_eig_opts()
    o.tol, o.maxit, o.inner_factor, o.inner_maxit = float(tol), int(maxit), float(inner_factor), int(inner_maxit)
    o.precond, o.loop = int(precond), int(loop)
    info = _abi.sla_eig_info()
    st = lib().sla_eig_smallest(ctypes.byref(_csr_struct(A)), _dev_ptr(v, dt, "v"), ctypes.byref(o),
                                ctypes.byref(info), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(dev))
    _check(st, "sla_eig_smallest")
    ei = EigInfo(int(info.iters), int(info.inner_iters), float(info.mu), float(info.residual), int(info.status))
    return ei.mu, v, ei


def sla_eig_grad_values(A: CSRMatrix, V: torch.Tensor, weights=None,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """grad_values[e] = sum_s w_s V[s, row(e)] V[s, col(e)] on A's pattern (V: [k, n] or [n]; asynchronous)."""
    dt, dev = A.values.dtype, A.values.device
    V2 = V.reshape(1, -1) if V.dim() == 1 else V
    k = int(V2.shape[0])
    if out is None:
        out = torch.empty(A.nnz, dtype=dt, device=dev)
    w = None
    if weights is not None:
        wl = [float(x) for x in weights]
        if len(wl) != k:
            raise ValueError("one weight per eigenvector")
        w = (ctypes.c_double * max(k, 1))(*wl)
    _check(lib().sla_eig_grad_values(ctypes.byref(_csr_struct(A)), k, _dev_ptr(V2, dt, "V") if k else None, w,
                                     _dev_ptr(out, dt, "grad_values"), _stream(dev)), "sla_eig_grad_values")
    return out


class EigSmallest(torch.autograd.Function):
    """(mu, v) = smallest eigenpair of SPD A; mu is differentiable with respect to A's values.

    Backward (Hellmann-Feynman): d mu / d values[e] = v[row(e)] * v[col(e)] on the pattern, so the
    node saves v and A only.  v is returned as a constant (no eigenvector gradient).
    """

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, tol, maxit, precond):
        A = CSRMatrix(row_ptr, col_idx, values)
        mu, v, info = sla_eig_smallest(A, tol=tol, maxit=maxit, precond=precond)
        if info.status == SLA_NOT_CONVERGED:
            warnings.warn(f"EigSmallest.forward: residual {info.residual:.3e} after {info.iters} steps")
        elif info.status != SLA_OK:
            raise SlaError(info.status, "EigSmallest.forward")
        ctx.save_for_backward(row_ptr, col_idx, values, v)
        ctx.mark_non_differentiable(v)
        return torch.tensor(mu, dtype=values.dtype, device=values.device), v

    @staticmethod
    def backward(ctx, g_mu, g_v):
        row_ptr, col_idx, values, v = ctx.saved_tensors
        if not ctx.needs_input_grad[2]:
            return None, None, None, None, None, None
        A = CSRMatrix(row_ptr, col_idx, values)
        gv = sla_eig_grad_values(A, v, weights=[float(g_mu)])
        return None, None, gv, None, None, None


def eigsh_smallest(A: CSRMatrix, tol: Optional[float] = None, maxit: int = 1000,
                   precond: int = SLA_PRECOND_NONE):
    """Differentiable smallest eigenvalue of SPD A (gradient to A.values) and its eigenvector."""
    return EigSmallest.apply(A.row_ptr, A.col_idx, A.values, tol, maxit, precond)


def sla_eigsh_workspace_bytes(n: int, k: int, dtype: torch.dtype, precond: int = SLA_PRECOND_NONE) -> int:
    return lib().sla_eigsh_workspace_bytes(int(n), int(k), _DT[dtype], int(precond))


def sla_eigsh(A: CSRMatrix, k: int, V0: Optional[torch.Tensor] = None, tol: Optional[float] = None,
              maxit: int = 2000, inner_factor: float = 0.01, inner_maxit: int = 100000,
              precond: int = SLA_PRECOND_NONE, loop: int = SLA_LOOP_AUTO, seed: int = 0,
              workspace: Optional[torch.Tensor] = None):
    """The k smallest eigenpairs of SPD A (1 <= k <= 16) by block inverse iteration with a
    Rayleigh-Ritz step.  Returns (mu [k] ascending, V [k, n] orthonormal rows, EigInfo).

    V0 ([k, n]) defaults to a block of standard normal entries drawn on the device from a generator
    seeded with `seed`; tol defaults to 1e-10 for float64 and 1e-5 for float32 data.
    """
    dt, dev = A.values.dtype, A.values.device
    if tol is None:
        tol = 1e-10 if dt == torch.float64 else 1e-5
    if V0 is None:
        gen = torch.Generator(device=dev)
        gen.manual_seed(int(seed))
        V = torch.randn(int(k), A.n, dtype=dt, device=dev, generator=gen)
    else:
        V = V0.detach().to(dtype=dt).contiguous().clone()
    if V.dim() != 2 or V.shape[0] != int(k) or V.shape[1] != A.n:
        raise ValueError("V0 must have shape [k, n]")
    need = sla_eigsh_workspace_bytes(A.n, k, dt, precond)
    ws = workspace if workspace is not None and workspace.numel() * workspace.element_size() >= need else \
        torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    o = _abi.sla_eig_opts()
    o.tol, o.maxit, o.inner_factor, o.inner_maxit = float(tol), int(maxit), float(inner_factor), int(inner_maxit)
    o.precond, o.loop = int(precond), int(loop)
    info = _abi.sla_eig_info()
    mu = (ctypes.c_double * int(k))()
    st = lib().sla_eigsh(ctypes.byref(_csr_struct(A)), int(k), _dev_ptr(V, dt, "V"), mu, ctypes.byref(o),
                         ctypes.byref(info), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(dev))
    _check(st, "sla_eigsh")
    ei = EigInfo(int(info.iters), int(info.inner_iters), float(info.mu), float(info.residual), int(info.status))
    return torch.tensor(list(mu), dtype=torch.float64), V, ei


class Eigsh(torch.autograd.Function):
    """(mu, V) = the k smallest eigenpairs of SPD A; mu ([k]) is differentiable with respect to A's
    values.  Backward (Hellmann-Feynman, summed over the pairs): d L / d values[e] =
    sum_s (dL/dmu_s) V[s, row(e)] V[s, col(e)] on the pattern.  Within a multiple eigenvalue only
    sums of gradients over the eigenspace are defined (L symmetric in its eigenvalues).  V is
    returned as a constant."""

    @staticmethod
    def forward(ctx, row_ptr, col_idx, values, k, tol, maxit, precond):
        A = CSRMatrix(row_ptr, col_idx, values)
        mu, V, info = sla_eigsh(A, k, tol=tol, maxit=maxit, precond=precond)
        if info.status == SLA_NOT_CONVERGED:
            warnings.warn(f"Eigsh.forward: largest residual {info.residual:.3e} after {info.iters} steps")
        elif info.status != SLA_OK:
            raise SlaError(info.status, "Eigsh.forward")
        ctx.save_for_backward(row_ptr, col_idx, values, V)
        ctx.mark_non_differentiable(V)
        return mu.to(dtype=values.dtype, device=values.device), V

    @staticmethod
    def backward(ctx, g_mu, g_V):
        row_ptr, col_idx, values, V = ctx.saved_tensors
        if not ctx.needs_input_grad[2]:
            return None, None, None, None, None, None, None
        A = CSRMatrix(row_ptr, col_idx, values)
        gv = sla_eig_grad_values(A, V, weights=[float(x) for x in g_mu.detach().cpu()])
        return None, None, gv, None, None, None, None


def eigsh(A: CSRMatrix, k: int = 1, tol: Optional[float] = None, maxit: int = 2000,
          precond: int = SLA_PRECOND_NONE):
    """Differentiable k smallest eigenvalues of SPD A ([k], ascending; gradient to A.values) and the
    eigenvectors ([k, n])."""
    return Eigsh.apply(A.row_ptr, A.col_idx, A.values, int(k), tol, maxit, precond)
