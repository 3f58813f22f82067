"""ctypes mirror of include/sla.h (structures, enums and prototypes of libsla)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsla.so")

SLA_OK, SLA_NOT_CONVERGED, SLA_BREAKDOWN, SLA_INVALID_ARG, SLA_BAD_CSR, SLA_NONFINITE = 0, 1, 2, 3, 4, 5
SLA_WORKSPACE_TOO_SMALL, SLA_TIMEOUT, SLA_CUDA_ERROR = 6, 7, 8
SLA_F32, SLA_F64 = 0, 1
SLA_I32, SLA_I64 = 0, 1
SLA_PRECOND_NONE, SLA_PRECOND_JACOBI = 0, 1
SLA_LOOP_AUTO, SLA_LOOP_HOST, SLA_LOOP_GRAPH, SLA_LOOP_RESIDENT, SLA_LOOP_CLUSTER = 0, 1, 2, 3, 4

# every symbol include/sla.h declares
EXPORTS = [
    "sla_status_string", "sla_last_cuda_error", "sla_version", "sla_launch_count", "sla_cg_workspace_bytes",
    "sla_validate_csr", "sla_spmv", "sla_cg_solve", "sla_cg_adjoint", "sla_grad_values", "sla_cg_solve_batched",
    "sla_cg_adjoint_batched", "sla_cg_solve_static", "sla_eig_workspace_bytes", "sla_eig_smallest",
    "sla_eig_grad_values", "sla_set_spmv_variant", "sla_test_set_barrier_wait", "sla_dist_state_bytes",
    "sla_dist_cg_begin", "sla_dist_cg_start", "sla_dist_cg_spmv", "sla_dist_cg_update", "sla_dist_cg_direction",
    "sla_dist_pack", "sla_dist_cg_info", "sla_spmv_transpose", "sla_matvec_grad_values", "sla_dist_scatter_add",
    "sla_graph_cache_stats", "sla_eigsh_workspace_bytes", "sla_eigsh", "sla_bicgstab_workspace_bytes",
    "sla_bicgstab_solve", "sla_bicgstab_adjoint",
]
SLA_SPMV_PLAIN, SLA_SPMV_TMA = 0, 1


class sla_csr(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("nnz", ctypes.c_int64), ("rowptr_type", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p),
                ("values", ctypes.c_void_p)]


class sla_cg_opts(ctypes.Structure):
    _fields_ = [("rtol", ctypes.c_double), ("maxit", ctypes.c_int64), ("precond", ctypes.c_int32),
                ("unroll", ctypes.c_int32), ("loop", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class sla_cg_info(ctypes.Structure):
    _fields_ = [("iters", ctypes.c_int64), ("rel_res", ctypes.c_double), ("status", ctypes.c_int32),
                ("path", ctypes.c_int32), ("kernels", ctypes.c_int64)]


class sla_eig_opts(ctypes.Structure):
    _fields_ = [("tol", ctypes.c_double), ("maxit", ctypes.c_int64), ("inner_factor", ctypes.c_double),
                ("inner_maxit", ctypes.c_int64), ("precond", ctypes.c_int32), ("loop", ctypes.c_int32)]


class sla_eig_info(ctypes.Structure):
    _fields_ = [("iters", ctypes.c_int64), ("inner_iters", ctypes.c_int64), ("mu", ctypes.c_double),
                ("residual", ctypes.c_double), ("status", ctypes.c_int32), ("pad", ctypes.c_int32)]


def bind(lib):
    P, C, O, I = ctypes.c_void_p, ctypes.POINTER(sla_csr), ctypes.POINTER(sla_cg_opts), ctypes.POINTER(sla_cg_info)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.sla_status_string.argtypes = [i32]
    lib.sla_status_string.restype = ctypes.c_char_p
    lib.sla_last_cuda_error.argtypes = []
    lib.sla_last_cuda_error.restype = ctypes.c_char_p
    lib.sla_version.argtypes = []
    lib.sla_version.restype = i32
    lib.sla_launch_count.argtypes = []
    lib.sla_launch_count.restype = ctypes.c_uint64
    lib.sla_cg_workspace_bytes.argtypes = [i64, i64, i32, i32]
    lib.sla_cg_workspace_bytes.restype = sz
    lib.sla_validate_csr.argtypes = [C, i32, ctypes.POINTER(i64), P, sz, P]
    lib.sla_spmv.argtypes = [C, P, P, P]
    lib.sla_cg_solve.argtypes = [C, P, P, O, P, I, P, P, sz, P]
    lib.sla_cg_adjoint.argtypes = [C, P, P, O, P, P, I, P, sz, P]
    lib.sla_grad_values.argtypes = [C, P, P, P, P]
    lib.sla_cg_solve_batched.argtypes = [C, i64, P, P, P, O, P, I, P, P, sz, P]
    lib.sla_cg_adjoint_batched.argtypes = [C, i64, P, P, P, O, P, P, I, P, sz, P]
    lib.sla_cg_solve_static.argtypes = [C, P, P, O, P, I, P, P]
    lib.sla_eig_workspace_bytes.argtypes = [i64, i32, i32]
    lib.sla_eig_workspace_bytes.restype = sz
    lib.sla_eig_smallest.argtypes = [C, P, ctypes.POINTER(sla_eig_opts), ctypes.POINTER(sla_eig_info), P, sz, P]
    lib.sla_eig_grad_values.argtypes = [C, i64, P, ctypes.POINTER(ctypes.c_double), P, P]
    lib.sla_bicgstab_workspace_bytes.argtypes = [i64, i64, i32]
    lib.sla_bicgstab_workspace_bytes.restype = sz
    lib.sla_bicgstab_solve.argtypes = [C, P, P, O, P, I, P, P, sz, P]
    lib.sla_bicgstab_adjoint.argtypes = [C, P, P, O, P, P, I, P, sz, P]
    lib.sla_eigsh_workspace_bytes.argtypes = [i64, i64, i32, i32]
    lib.sla_eigsh_workspace_bytes.restype = sz
    lib.sla_eigsh.argtypes = [C, i64, P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(sla_eig_opts),
                              ctypes.POINTER(sla_eig_info), P, sz, P]
    lib.sla_spmv_transpose.argtypes = [C, P, P, P, P]
    lib.sla_matvec_grad_values.argtypes = [C, P, P, P, P]
    lib.sla_dist_scatter_add.argtypes = [i64, i32, P, P, i64, P, P]
    lib.sla_dist_state_bytes.argtypes = []
    lib.sla_dist_state_bytes.restype = sz
    lib.sla_dist_cg_begin.argtypes = [C, i64, P, O, P, P, P, P, P, P, P, P]
    lib.sla_dist_cg_start.argtypes = [P, i32, P, P, P]
    lib.sla_dist_cg_spmv.argtypes = [C, i64, P, P, P, P, P]
    lib.sla_dist_cg_update.argtypes = [i64, i32, i32, P, i32, P, P, P, P, P, P, P, P, P]
    lib.sla_dist_cg_direction.argtypes = [i64, i32, P, i32, P, P, P, P, P]
    lib.sla_dist_pack.argtypes = [i64, i32, P, P, i64, P, P]
    lib.sla_dist_cg_info.argtypes = [P, I, ctypes.POINTER(i32), P]
    lib.sla_set_spmv_variant.argtypes = [i32]
    lib.sla_graph_cache_stats.argtypes = [ctypes.POINTER(i64)] * 3
    lib.sla_test_set_barrier_wait.argtypes = [ctypes.c_uint32, i64]
    for name in ["sla_spmv_transpose", "sla_matvec_grad_values", "sla_dist_scatter_add", "sla_dist_cg_begin", "sla_dist_cg_start", "sla_dist_cg_spmv", "sla_dist_cg_update",
                 "sla_dist_cg_direction", "sla_dist_pack", "sla_dist_cg_info",
                 "sla_set_spmv_variant", "sla_graph_cache_stats", "sla_test_set_barrier_wait", "sla_validate_csr", "sla_spmv", "sla_cg_solve", "sla_cg_adjoint", "sla_grad_values",
                 "sla_cg_solve_batched", "sla_cg_adjoint_batched", "sla_cg_solve_static", "sla_eig_smallest",
                 "sla_eig_grad_values", "sla_eigsh", "sla_bicgstab_solve", "sla_bicgstab_adjoint"]:
        getattr(lib, name).restype = i32
    return lib


def load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise RuntimeError(f"libsla is not built ({path} missing): run differentiable_sparse_iterative_gb300/build.py "
                           "or __graft_entry__.build(); there is no fallback implementation")
    return bind(ctypes.CDLL(path))
