"""A host (numpy) stand-in for libsla's distributed steps, for the CPU tests of the distributed layer.

TEST INFRASTRUCTURE ONLY.  The product runs these steps as libsla kernels
(differentiable_sparse_iterative_gb300.distributed.LibslaOps, CUDA tensors only).  The gloo tests on
CPU ranks use this stand-in instead, so that the host logic of the distributed layer -- row
partition, local blocks, exchange plan, halo exchange, gathering of partials in rank order, the
shared stopping decision -- runs over real process groups without a GPU.  Each method follows the
contract of the libsla call of the same name in include/sla.h (sla_dist_cg_begin, ...), on torch
CPU tensors, with the textbook Hestenes-Stiefel recurrences.
"""
from types import SimpleNamespace

import numpy as np

OK, NOT_CONVERGED, BREAKDOWN, NONFINITE = 0, 1, 2, 5


def _a(t):
    return None if t is None else t.numpy()


def _local_spmv(A, n_own, v):
    """Owned rows of A_ext v, each row summed in storage order (one entry position at a time)."""
    rp, ci, val = A.row_ptr.numpy().astype(np.int64), A.col_idx.numpy(), A.values.numpy()
    lens = np.diff(rp[: n_own + 1])
    out = np.zeros(n_own, dtype=val.dtype)
    for k in range(int(lens.max()) if n_own else 0):
        rows = np.nonzero(lens > k)[0]
        e = rp[rows] + k
        out[rows] = out[rows] + val[e] * v[ci[e]]
    return out


class NumpyOps:
    def state(self, device):
        return {"done": 1, "status": NOT_CONVERGED, "k": 0, "rel_res": 0.0}

    def begin(self, A, n_own, b, opts, x, r, z, p_ext, dinv, part5, S, stream):
        S.clear()
        S.update(rtol=opts.rtol, maxit=opts.maxit, precond=opts.precond, done=1, status=NOT_CONVERGED, k=0,
                 rel_res=0.0, alpha=0.0, beta=0.0)
        bn = _a(b)[:n_own]
        _a(x)[:n_own] = 0.0
        _a(r)[:n_own] = bn
        parts = [float(bn @ bn), float(bn @ bn), 0.0, 0.0, 0.0]
        zz = bn
        if opts.precond == 1:
            rp, ci, val = A.row_ptr.numpy().astype(np.int64), A.col_idx.numpy(), A.values.numpy()
            d = np.zeros(n_own)
            for i in range(n_own):
                for e in range(rp[i], rp[i + 1]):
                    if ci[e] == i:
                        d[i] = val[e]
            parts[3] = float(np.sum(~np.isfinite(d)))
            parts[4] = float(np.sum(np.isfinite(d) & ~(d > 0)))
            with np.errstate(divide="ignore", invalid="ignore"):
                di = 1.0 / d
            _a(dinv)[:n_own] = di
            zz = di * bn
            _a(z)[:n_own] = zz
            parts[2] = float(bn @ zz)
        _a(p_ext)[:n_own] = zz
        _a(part5)[:] = parts

    def start(self, g, R, S, history, stream):
        g = _a(g).reshape(R, 5)
        bb = rr = rz = nf = npos = 0.0
        for q in range(R):
            bb += g[q, 0]; rr += g[q, 1]; rz += g[q, 2]; nf += g[q, 3]; npos += g[q, 4]  # noqa: E702
        nb = np.sqrt(bb)
        S["nb"], S["k"], S["done"] = nb, 0, 1
        jac = S["precond"] == 1
        if not np.isfinite(nb):
            S["status"] = NONFINITE
        elif nb == 0.0:
            S["status"] = OK
            if history is not None:
                _a(history)[0] = 0.0
        elif jac and nf > 0:
            S["status"] = NONFINITE
        elif jac and npos > 0:
            S["status"] = BREAKDOWN
        else:
            S["rel_res"] = np.sqrt(rr) / nb
            if history is not None:
                _a(history)[0] = S["rel_res"]
            if not np.isfinite(rr):
                S["status"] = NONFINITE
            elif np.sqrt(rr) <= S["rtol"] * nb:
                S["status"] = OK
            elif S["maxit"] == 0:
                S["status"] = NOT_CONVERGED
            else:
                S["done"] = 0
                S["rho"] = rz if jac else rr
                S["tol"] = S["rtol"] * nb

    def spmv(self, A, n_own, p_ext, q, part1, S, stream):
        if S["done"]:
            return
        qq = _local_spmv(A, n_own, _a(p_ext))
        _a(q)[:n_own] = qq
        _a(part1)[0] = float(_a(p_ext)[:n_own] @ qq)

    def update(self, n_own, dtype, precond, g, R, x, r, p_ext, q, dinv, z, part2, S, stream):
        if S["done"]:
            return
        pq = 0.0
        for v in _a(g)[:R]:
            pq += v
        if not np.isfinite(pq) or not pq > 0.0:
            S["status"], S["done"] = (NONFINITE if not np.isfinite(pq) else BREAKDOWN), 1
            _a(part2)[:] = 0.0
            return
        al = S["rho"] / pq
        S["alpha"] = al
        xa, ra, pa, qa = _a(x), _a(r), _a(p_ext), _a(q)
        xa[:n_own] = xa[:n_own] + al * pa[:n_own]
        ra[:n_own] = ra[:n_own] - al * qa[:n_own]
        rr = float(ra[:n_own] @ ra[:n_own])
        rz = 0.0
        if precond == 1:
            _a(z)[:n_own] = _a(dinv)[:n_own] * ra[:n_own]
            rz = float(ra[:n_own] @ _a(z)[:n_own])
        _a(part2)[:] = [rr, rz]

    def direction(self, n_own, dtype, g, R, zr, p_ext, history, S, stream):
        if S["done"]:
            return
        g = _a(g).reshape(R, 2)
        rr = rz = 0.0
        for q in range(R):
            rr += g[q, 0]
            rz += g[q, 1]
        if S["precond"] != 1:
            rz = rr
        k = S["k"] + 1
        S["k"] = k
        S["rel_res"] = np.sqrt(rr) / S["nb"]
        if history is not None:
            _a(history)[k] = S["rel_res"]
        if not np.isfinite(rr):
            S["status"], S["done"] = NONFINITE, 1
        elif np.sqrt(rr) <= S["tol"]:
            S["status"], S["done"] = OK, 1
        elif k >= S["maxit"]:
            S["status"], S["done"] = NOT_CONVERGED, 1
        else:
            beta = rz / S["rho"]
            S["beta"], S["rho"] = beta, rz
            pa = _a(p_ext)
            pa[:n_own] = _a(zr)[:n_own] + beta * pa[:n_own]

    def pack(self, n, dtype, v, idx, buf, stream):
        _a(buf)[:] = _a(v)[_a(idx)]

    def info(self, S, stream):
        return SimpleNamespace(iters=S["k"], rel_res=S["rel_res"], status=S["status"]), S["done"]

    def product(self, A, x, y, stream):
        n = A.row_ptr.shape[0] - 1
        _a(y)[:] = _local_spmv(A, n, _a(x))

    def scatter_add(self, n, dtype, v, idx, buf, stream):
        va, ia, ba = _a(v), _a(idx), _a(buf)
        for t in range(ia.shape[0]):
            if 0 <= ia[t] < n:
                va[ia[t]] += ba[t]

    def matvec_grad(self, A, gy, x, gv, stream):
        rp, ci = A.row_ptr.numpy().astype(np.int64), A.col_idx.numpy()
        rows = np.repeat(np.arange(A.row_ptr.shape[0] - 1), np.diff(rp))
        _a(gv)[:] = _a(gy)[rows] * _a(x)[ci]

    def grad_values(self, A, lam_ext, x_ext, gv, stream):
        rp, ci = A.row_ptr.numpy().astype(np.int64), A.col_idx.numpy()
        rows = np.repeat(np.arange(A.row_ptr.shape[0] - 1), np.diff(rp))
        _a(gv)[:] = -(_a(lam_ext)[rows] * _a(x_ext)[ci])
