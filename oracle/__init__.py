"""fp64 CPU oracle for the differentiable CSR conjugate-gradient solve (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The oracle is the checker that the CUDA library is
compared against; it is loaded only by the test suite, by the smoke check and
by the benchmark's CPU-baseline leg, never by the library itself.  It shares no
code with the CUDA path.

Each function follows "torch-sla: Differentiable Sparse Linear Algebra with
Adjoint Solvers and Sparse Tensor Parallelism for PyTorch" (Chi, Wen),
technical summary, Methodology sections 1 (native iterative solver, .matvec /
.solve) and 2 (adjoint differentiation framework: linear systems, and the
eigenvalue gradient v_i v_j on the pattern); see the C source ``sla_oracle.c``
for the readings taken where the pages are silent.

Parity pins live in ``tests/test_oracle_*.py``.  Every oracle function is
pinned there against something other than itself (dense linear algebra on
tiny grids, closed-form eigenvalues and CG bounds, finite termination, the
adjoint identity, central finite differences, exact scaling invariants, the
closed-form fundamental mode of the five-point Laplacian).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LIB_OMP_PATH = os.path.join(_HERE, "liboracle_omp.so")
_lib = None
_lib_omp = None

STATUS = {0: "OK", 1: "NOT_CONVERGED", 2: "BREAKDOWN", 5: "NONFINITE"}


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, openmp: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -ffp-contract=off: no fused multiply-add).

    openmp=True makes the multi-core build of the same file (chunked dot products whose result
    does not depend on the thread count; see the C source's header)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        flags = ["-fopenmp"] if openmp else []
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", *flags,
                        "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> None:
    """Both builds: the plain one-thread library and the multi-core one."""
    build(force)
    build(force, out=_LIB_OMP_PATH, openmp=True)


def _bind(lib):
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.orc_spmv.argtypes = [i64, p, p, p, p, p]
    lib.orc_spmv.restype = None
    lib.orc_dot.argtypes = [i64, p, p]
    lib.orc_dot.restype = ctypes.c_double
    lib.orc_diagonal.argtypes = [i64, p, p, p, p]
    lib.orc_diagonal.restype = None
    lib.orc_cg.argtypes = [i64, p, p, p, p, p, ctypes.c_double, i64, ctypes.c_int, p, p,
                           ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
    lib.orc_cg.restype = ctypes.c_int
    lib.orc_grad_values.argtypes = [i64, p, p, p, p, p]
    lib.orc_grad_values.restype = None
    lib.orc_cg_adjoint.argtypes = [i64, p, p, p, p, p, ctypes.c_double, i64, ctypes.c_int, p, p,
                                   ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
    lib.orc_cg_adjoint.restype = ctypes.c_int
    lib.orc_eig_grad_values.argtypes = [i64, p, p, i64, p, p, p]
    lib.orc_eig_grad_values.restype = None
    lib.orc_spmv_transpose.argtypes = [i64, p, p, p, p, p]
    lib.orc_spmv_transpose.restype = None
    lib.orc_matvec_grad_values.argtypes = [i64, p, p, p, p, p]
    lib.orc_matvec_grad_values.restype = None
    lib.orc_threads.argtypes = [ctypes.c_int]
    lib.orc_threads.restype = ctypes.c_int
    lib.orc_transpose.argtypes = [i64, p, p, p, p, p, p]
    lib.orc_transpose.restype = None
    lib.orc_bicgstab.argtypes = [i64, p, p, p, p, p, ctypes.c_double, i64, p, p, ctypes.POINTER(i64),
                                 ctypes.POINTER(ctypes.c_double)]
    lib.orc_bicgstab.restype = ctypes.c_int
    lib.orc_bicgstab_adjoint.argtypes = [i64, p, p, p, p, p, ctypes.c_double, i64, p, p, ctypes.POINTER(i64),
                                         ctypes.POINTER(ctypes.c_double)]
    lib.orc_bicgstab_adjoint.restype = ctypes.c_int
    return lib


def load(path: Optional[str] = None):
    """Load (building if needed) the plain one-thread oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - not Linux
        return os.cpu_count() or 1


def load_parallel(threads: Optional[int] = None):
    """Load (building if needed) the multi-core oracle library; threads defaults to every host core.

    Its results do not depend on the thread count; they differ from the plain build's only by
    the dot products' summation order (fixed chunks)."""
    global _lib_omp
    if _lib_omp is None:
        _lib_omp = _bind(ctypes.CDLL(build(out=_LIB_OMP_PATH, openmp=True)))
    _lib_omp.orc_threads(int(threads) if threads else host_cores())
    return _lib_omp


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _csr(row_ptr, col_idx, values):
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    v = np.ascontiguousarray(values, dtype=np.float64)
    return rp, ci, v


def spmv(row_ptr, col_idx, values, x, lib=None) -> np.ndarray:
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(n, dtype=np.float64)
    lib.orc_spmv(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(x), _ptr(y))
    return y


def spmv_transpose(row_ptr, col_idx, values, x, lib=None) -> np.ndarray:
    """y = A^T x (square A)."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(n, dtype=np.float64)
    lib.orc_spmv_transpose(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(x), _ptr(y))
    return y


def matvec_grad_values(row_ptr, col_idx, gy, x, lib=None) -> np.ndarray:
    """grad_values[k] = gy[row(k)] * x[col(k)]: the gradient of L(A x) with respect to the stored values."""
    lib = lib or load()
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = rp.shape[0] - 1
    gy = np.ascontiguousarray(gy, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    gv = np.empty(ci.shape[0], dtype=np.float64)
    lib.orc_matvec_grad_values(n, _ptr(rp), _ptr(ci), _ptr(gy), _ptr(x), _ptr(gv))
    return gv


def dot(a, b, lib=None) -> float:
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    return float(lib.orc_dot(a.shape[0], _ptr(a), _ptr(b)))


def cg(row_ptr, col_idx, values, b, x0=None, rtol: float = 1e-10, maxit: int = 100000, precond: int = 0,
       history: bool = False, lib=None) -> dict:
    """Solve A x = b by CG; returns dict(x, iters, rel_res, status, history)."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    b = np.ascontiguousarray(b, dtype=np.float64)
    x0c = None if x0 is None else np.ascontiguousarray(x0, dtype=np.float64)
    x = np.empty(n, dtype=np.float64)
    h = np.full(maxit + 1, np.nan) if history else None
    it = ctypes.c_int64(0)
    rr = ctypes.c_double(0.0)
    st = lib.orc_cg(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(b), _ptr(x0c), float(rtol), int(maxit), int(precond),
                    _ptr(x), _ptr(h), ctypes.byref(it), ctypes.byref(rr))
    out = {"x": x, "iters": int(it.value), "rel_res": float(rr.value), "status": int(st)}
    if history:
        out["history"] = h[: it.value + 1].copy()
    return out


def grad_values(row_ptr, col_idx, lam, x, lib=None) -> np.ndarray:
    lib = lib or load()
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = rp.shape[0] - 1
    lam = np.ascontiguousarray(lam, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    gv = np.empty(ci.shape[0], dtype=np.float64)
    lib.orc_grad_values(n, _ptr(rp), _ptr(ci), _ptr(lam), _ptr(x), _ptr(gv))
    return gv


def cg_adjoint(row_ptr, col_idx, values, x, g, rtol: float = 1e-10, maxit: int = 100000, precond: int = 0,
               lib=None) -> dict:
    """Adjoint backward: dict(grad_b = lambda, grad_values, iters, rel_res, status)."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    gb = np.empty(n, dtype=np.float64)
    gv = np.empty(ci.shape[0], dtype=np.float64)
    it = ctypes.c_int64(0)
    rr = ctypes.c_double(0.0)
    st = lib.orc_cg_adjoint(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(x), _ptr(g), float(rtol), int(maxit),
                            int(precond), _ptr(gb), _ptr(gv), ctypes.byref(it), ctypes.byref(rr))
    return {"grad_b": gb, "grad_values": gv, "iters": int(it.value), "rel_res": float(rr.value),
            "status": int(st)}


def transpose(row_ptr, col_idx, values, lib=None):
    """A^T as CSR (row_ptr int64, col_idx int32, values): each column's entries in increasing row order."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    trp = np.empty(n + 1, dtype=np.int64)
    tci = np.empty(ci.shape[0], dtype=np.int32)
    tv = np.empty(ci.shape[0], dtype=np.float64)
    lib.orc_transpose(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(trp), _ptr(tci), _ptr(tv))
    return trp, tci, tv


def bicgstab(row_ptr, col_idx, values, b, x0=None, rtol: float = 1e-10, maxit: int = 100000,
             history: bool = False, lib=None) -> dict:
    """Solve a general A x = b by BiCGStab; returns dict(x, iters, rel_res, status, history)."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    b = np.ascontiguousarray(b, dtype=np.float64)
    x0c = None if x0 is None else np.ascontiguousarray(x0, dtype=np.float64)
    x = np.empty(n, dtype=np.float64)
    h = np.full(maxit + 1, np.nan) if history else None
    it = ctypes.c_int64(0)
    rr = ctypes.c_double(0.0)
    st = lib.orc_bicgstab(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(b), _ptr(x0c), float(rtol), int(maxit), _ptr(x),
                          _ptr(h), ctypes.byref(it), ctypes.byref(rr))
    out = {"x": x, "iters": int(it.value), "rel_res": float(rr.value), "status": int(st)}
    if history:
        out["history"] = h[: it.value + 1].copy()
    return out


def bicgstab_adjoint(row_ptr, col_idx, values, x, g, rtol: float = 1e-10, maxit: int = 100000, lib=None) -> dict:
    """Adjoint backward of the BiCGStab solve: dict(grad_b = lambda (A^T lambda = g), grad_values, iters,
    rel_res, status)."""
    lib = lib or load()
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    gb = np.empty(n, dtype=np.float64)
    gv = np.empty(ci.shape[0], dtype=np.float64)
    it = ctypes.c_int64(0)
    rr = ctypes.c_double(0.0)
    st = lib.orc_bicgstab_adjoint(n, _ptr(rp), _ptr(ci), _ptr(v), _ptr(x), _ptr(g), float(rtol), int(maxit),
                                  _ptr(gb), _ptr(gv), ctypes.byref(it), ctypes.byref(rr))
    return {"grad_b": gb, "grad_values": gv, "iters": int(it.value), "rel_res": float(rr.value),
            "status": int(st)}


def cg_batched(row_ptr, col_idx, values_b, b_b, rtol, maxit, precond=0, history=False, lib=None) -> list:
    """Batched shared-pattern solve: one fp64 CG per system on the (possibly fp32-rounded) inputs."""
    return [cg(row_ptr, col_idx, values_b[s], b_b[s], None, rtol, maxit, precond, history, lib)
            for s in range(values_b.shape[0])]


def cg_adjoint_batched(row_ptr, col_idx, values_b, x_b, g_b, rtol, maxit, precond=0, lib=None) -> list:
    return [cg_adjoint(row_ptr, col_idx, values_b[s], x_b[s], g_b[s], rtol, maxit, precond, lib)
            for s in range(values_b.shape[0])]


# --------------------------------------------------------------------------- eigenvalue problems
#
# Methodology 2, eigenvalue problems: the gradient of an eigenvalue with respect to the matrix is
# v_i v_j on the sparsity pattern (Hellmann-Feynman).  The eigenpair itself has a plain
# definition, so the oracle takes it from a dense symmetric eigensolver (numpy.linalg.eigh) on
# small matrices; how the GPU reaches it (inverse iteration) does not enter the oracle.

def dense(row_ptr, col_idx, values) -> np.ndarray:
    """The CSR matrix as a dense fp64 array (small n only)."""
    rp, ci, v = _csr(row_ptr, col_idx, values)
    n = rp.shape[0] - 1
    D = np.zeros((n, n))
    for i in range(n):
        for e in range(rp[i], rp[i + 1]):
            D[i, ci[e]] += v[e]
    return D


def sign_normalise(v: np.ndarray) -> np.ndarray:
    """The eigenvector's sign: the sum of its entries is made >= 0 (ties: the first nonzero entry > 0)."""
    s = float(np.sum(v))
    if s < 0.0 or (s == 0.0 and v[np.flatnonzero(v)[0]] < 0.0):
        return -v
    return v


def eig_smallest(row_ptr, col_idx, values, k: int = 1):
    """The k smallest eigenvalues (ascending) and unit eigenvectors [k, n] of symmetric A (dense eigh)."""
    D = dense(row_ptr, col_idx, values)
    if not np.array_equal(D, D.T):
        raise ValueError("eig_smallest needs a symmetric matrix")
    mu, U = np.linalg.eigh(D)
    V = np.stack([sign_normalise(U[:, s]) for s in range(k)])
    return mu[:k].copy(), V


def eig_grad_values(row_ptr, col_idx, V, w=None, lib=None) -> np.ndarray:
    """grad_values[e] = sum_s (w_s v_s[i]) v_s[j] on A's pattern (V: [k, n]; w: k weights or None = ones)."""
    lib = lib or load()
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = rp.shape[0] - 1
    V = np.ascontiguousarray(np.atleast_2d(V), dtype=np.float64)
    k = V.shape[0] if V.size else 0
    wc = None if w is None else np.ascontiguousarray(w, dtype=np.float64)
    if wc is not None and wc.shape[0] != k:
        raise ValueError("one weight per eigenvector")
    gv = np.empty(ci.shape[0], dtype=np.float64)
    lib.orc_eig_grad_values(n, _ptr(rp), _ptr(ci), k, _ptr(V), _ptr(wc), _ptr(gv))
    return gv
