"""Coefficient-to-matrix map for the gradient-through-the-solve tests.

The Dirichlet diffusion matrix of workloads.diffusion_dirichlet is linear in its 2m(m+1) edge
conductivities k: values = M k for a fixed sparse M (nnz x edges).  M is recovered column by
column from the generator itself (values of a unit conductivity on one edge), so the tests
do not restate the assembly.
"""
import numpy as np

from workloads import diffusion_dirichlet


def edge_map(m: int):
    """(pattern CSR, rows, cols, weights) of M in COO form: values[rows] += weights * k[cols]."""
    E = 2 * m * (m + 1)
    base = diffusion_dirichlet(m, np.zeros(E))
    rows, cols, wts = [], [], []
    for j in range(E):
        e = np.zeros(E)
        e[j] = 1.0
        v = diffusion_dirichlet(m, e).values
        nz = np.nonzero(v)[0]
        rows.append(nz)
        cols.append(np.full(nz.size, j))
        wts.append(v[nz])
    return base, np.concatenate(rows), np.concatenate(cols), np.concatenate(wts)


def apply_map(nnz: int, rows, cols, wts, k):
    out = np.zeros(nnz)
    np.add.at(out, rows, wts * k[cols])
    return out


def apply_map_t(E: int, rows, cols, wts, gv):
    out = np.zeros(E)
    np.add.at(out, cols, wts * gv[rows])
    return out
