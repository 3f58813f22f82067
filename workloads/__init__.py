"""Seeded synthetic inputs for the CSR conjugate-gradient solve and its adjoint.

This module is shared by the oracle's tests, the GPU parity tests and the
benchmark.  It holds the random draws and the assembly of the test matrices
(2D five-point Poisson and variable-coefficient diffusion on a grid), and none
of the solver's arithmetic: no dot product and no conjugate-gradient step.  The
one product with a matrix it evaluates is input generation, the same on both
sides: the manufactured right-hand side b = A x* of the 64 x 64 Poisson
workload, taken on the grid by the five-point stencil (``_stencil_apply``)
rather than through a CSR product.

Workloads follow the experiments of "torch-sla: Differentiable Sparse Linear
Algebra with Adjoint Solvers and Sparse Tensor Parallelism for PyTorch"
(Chi, Wen), technical summary, section "Experimental Results" (2D Poisson
benchmarks; 1M DOF; 169M DOF on one GPU) and the limitation noted under
"Significance" (Jacobi preconditioning for the PyTorch-native backend).  The
pages name no dataset: every input is synthetic.

Conventions (all generators):
  * unknowns are numbered row-major on an m x m interior grid, i = a*m + c;
  * CSR columns are sorted ascending within each row; the diagonal is stored;
  * col_idx is int32; row_ptr is int32 unless ``rowptr64`` is requested;
  * values are float64 (float32 copies are made by rounding the float64 ones);
  * "log-normal(mu, sigma)" means exp(N(mu, sigma^2)) as drawn by
    ``numpy.random.Generator.lognormal``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "CSR", "poisson_5pt", "diffusion_interior", "diffusion_dirichlet",
    "random_spd", "Workload", "config1", "config2", "config3", "config4", "config5",
    "small_poisson", "config_by_name",
]


@dataclass
class CSR:
    n: int
    row_ptr: np.ndarray  # int32 or int64, n+1
    col_idx: np.ndarray  # int32, nnz
    values: np.ndarray   # float64 (or float32), nnz

    @property
    def nnz(self) -> int:
        return int(self.col_idx.shape[0])

    def astype(self, dtype) -> "CSR":
        return CSR(self.n, self.row_ptr, self.col_idx, self.values.astype(dtype))

    def dense(self) -> np.ndarray:
        """Dense copy (only for tiny matrices in tests)."""
        A = np.zeros((self.n, self.n), dtype=np.float64)
        rows = np.repeat(np.arange(self.n), np.diff(self.row_ptr.astype(np.int64)))
        A[rows, self.col_idx.astype(np.int64)] = self.values
        return A


def _pattern_5pt(m: int, rowptr64: bool, chunk_rows: int = 1 << 22):
    """Five-point pattern on an m x m grid, Dirichlet: missing neighbours dropped.

    Returns (row_ptr, col_idx, slot) where slot[k] in {0..4} says which stencil
    position entry k is (0: north i-m, 1: west i-1, 2: centre, 3: east i+1,
    4: south i+m).  Built in chunks of grid rows to bound host memory.
    """
    n = m * m
    a = np.arange(m, dtype=np.int64)
    cnt_row = 5 - (a == 0) - (a == m - 1)          # per grid row, before west/east
    # count per unknown = 5 - [a==0] - [a==m-1] - [c==0] - [c==m-1]; for m == 1 the
    # centre alone remains.
    c = np.arange(m, dtype=np.int64)
    cnt_col = -(c == 0).astype(np.int64) - (c == m - 1).astype(np.int64)
    counts = (cnt_row[:, None] + cnt_col[None, :]).reshape(-1)
    if m == 1:
        counts = np.ones(1, dtype=np.int64)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    nnz = int(row_ptr[-1])
    col_idx = np.empty(nnz, dtype=np.int32)
    slot = np.empty(nnz, dtype=np.int8)
    offs = np.array([-m, -1, 0, 1, m], dtype=np.int64)
    rows_per_chunk = max(1, chunk_rows // m)
    for a0 in range(0, m, rows_per_chunk):
        a1 = min(m, a0 + rows_per_chunk)
        aa = np.repeat(np.arange(a0, a1, dtype=np.int64), m)
        cc = np.tile(np.arange(m, dtype=np.int64), a1 - a0)
        i = aa * m + cc
        cand = i[:, None] + offs[None, :]
        valid = np.stack([aa > 0, cc > 0, np.ones_like(aa, dtype=bool), cc < m - 1, aa < m - 1], axis=1)
        k0, k1 = int(row_ptr[a0 * m]), int(row_ptr[a1 * m])
        col_idx[k0:k1] = cand[valid]
        slot[k0:k1] = np.broadcast_to(np.arange(5, dtype=np.int8), cand.shape)[valid]
    rp = row_ptr if rowptr64 else row_ptr.astype(np.int32)
    return rp, col_idx, slot


def poisson_5pt(m: int, rowptr64: bool = False) -> CSR:
    """2D Poisson five-point Laplacian, diagonal 4, neighbours -1, no h^2 scaling.

    nnz = 5 m^2 - 4 m.  Eigenvalues 4 - 2cos(i pi/(m+1)) - 2cos(j pi/(m+1)).
    """
    rp, ci, slot = _pattern_5pt(m, rowptr64)
    vals = np.where(slot == 2, 4.0, -1.0)
    return CSR(m * m, rp, ci, vals)


def convection_diffusion(m: int, cx: float = 0.4, cy: float = 0.25, rowptr64: bool = False) -> CSR:
    """2D convection-diffusion on the five-point pattern, central differences: diagonal 4, west
    -1 - cx, east -1 + cx, north (i - m) -1 - cy, south (i + m) -1 + cy, missing neighbours dropped.

    Non-symmetric (for cx or cy nonzero) on a structurally symmetric pattern; for |cx|, |cy| < 1
    every off-diagonal entry is negative and each row sums to at least 0, so it is a nonsingular
    M-matrix.  The input of the non-symmetric (BiCGStab) path.
    """
    rp, ci, slot = _pattern_5pt(m, rowptr64)
    off = np.array([-1.0 - cy, -1.0 - cx, 4.0, -1.0 + cx, -1.0 + cy])
    return CSR(m * m, rp, ci, off[slot.astype(np.int64)])


def _edge_values(m: int, slot: np.ndarray, rp: np.ndarray, kN, kW, kE, kS, shift: float) -> np.ndarray:
    """Fill CSR values from per-unknown edge conductivities (each an m x m array).

    Off-diagonal to the north neighbour is -kN, to the west -kW, east -kE,
    south -kS.  The diagonal is ((((kN + kW) + kE) + kS) + shift) with absent
    edges given as 0; the order is fixed so the values are reproducible.
    """
    n = m * m
    rows = np.repeat(np.arange(n, dtype=np.int64), np.diff(rp.astype(np.int64)))
    diag = (((kN + kW) + kE) + kS) + shift
    stacks = [kN.reshape(-1), kW.reshape(-1), None, kE.reshape(-1), kS.reshape(-1)]
    vals = np.empty(slot.shape[0], dtype=np.float64)
    for s in range(5):
        sel = slot == s
        if s == 2:
            vals[sel] = diag.reshape(-1)[rows[sel]]
        else:
            vals[sel] = -stacks[s][rows[sel]]
    return vals


def diffusion_interior(m: int, k: np.ndarray, shift: float) -> CSR:
    """Weighted graph Laplacian of the m x m grid over its 2m(m-1) interior edges, plus shift*I.

    ``k`` holds the edge conductivities: first the m(m-1) horizontal edges
    (a,c)-(a,c+1), row-major in (a, c); then the (m-1)m vertical edges
    (a,c)-(a+1,c), row-major in (a, c).  Every row sums to ``shift``.
    """
    k = np.asarray(k, dtype=np.float64)
    assert k.shape == (2 * m * (m - 1),)
    h = k[: m * (m - 1)].reshape(m, m - 1)
    v = k[m * (m - 1):].reshape(m - 1, m)
    kN = np.zeros((m, m)); kS = np.zeros((m, m)); kW = np.zeros((m, m)); kE = np.zeros((m, m))
    kW[:, 1:] = h; kE[:, :-1] = h
    kN[1:, :] = v; kS[:-1, :] = v
    rp, ci, slot = _pattern_5pt(m, False)
    return CSR(m * m, rp, ci, _edge_values(m, slot, rp, kN, kW, kE, kS, shift))


def diffusion_dirichlet(m: int, k: np.ndarray, rowptr64: bool = False) -> CSR:
    """Variable-coefficient diffusion with Dirichlet boundary edges, 2m(m+1) edges in all.

    ``k``: first the m(m+1) horizontal edges h[a, c], c = 0..m, between
    (a, c-1) and (a, c) (c = 0 and c = m touch the boundary); then the (m+1)m
    vertical edges v[a, c], a = 0..m, between (a-1, c) and (a, c).  A boundary
    edge adds its conductivity to the diagonal only.  With every k = 1 this is
    exactly the Poisson matrix of ``poisson_5pt``.
    """
    k = np.asarray(k, dtype=np.float64)
    assert k.shape == (2 * m * (m + 1),)
    h = k[: m * (m + 1)].reshape(m, m + 1)
    v = k[m * (m + 1):].reshape(m + 1, m)
    kW = h[:, :-1]; kE = h[:, 1:]; kN = v[:-1, :]; kS = v[1:, :]
    rp, ci, slot = _pattern_5pt(m, rowptr64)
    return CSR(m * m, rp, ci, _edge_values(m, slot, rp, kN, kW, kE, kS, 0.0))


def banded_dominant(n: int, half_band: int, chunk_rows: int = 1 << 16) -> CSR:
    """Symmetric banded matrix with int64 row_ptr: row i stores columns max(0, i - h) .. min(n - 1,
    i + h) in increasing order, -1 off the diagonal and (number of off-diagonal entries + 1) on it,
    so it is strictly diagonally dominant, hence SPD.  Built in row chunks straight into the final
    arrays, so that a pattern with more than 2^31 entries (the 64-bit row-offset case) costs its
    own size in host memory and little more."""
    h = int(half_band)
    i = np.arange(n, dtype=np.int64)
    lens = np.minimum(i, h) + np.minimum(n - 1 - i, h) + 1
    rp = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(lens, out=rp[1:])
    nnz = int(rp[-1])
    ci = np.empty(nnz, dtype=np.int32)
    vals = np.full(nnz, -1.0)
    offs = np.arange(-h, h + 1, dtype=np.int64)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        cols = np.arange(r0, r1, dtype=np.int64)[:, None] + offs[None, :]
        keep = (cols >= 0) & (cols < n)
        ci[rp[r0]:rp[r1]] = cols[keep].astype(np.int32)
        diag = rp[r0:r1] + np.minimum(np.arange(r0, r1), h)  # position of (i, i) in row i
        vals[diag] = lens[r0:r1].astype(np.float64)  # off-diagonal count + 1
    return CSR(n, rp, ci, vals)


def random_spd(n: int, avg_offdiag: float, seed: int, long_rows: int = 0, shift: float = 1.0) -> CSR:
    """Random symmetric strictly diagonally dominant (hence SPD) CSR matrix.

    Off-diagonal pairs (i, j) are drawn uniformly with weights w ~ U(0.1, 1);
    ``long_rows`` rows are additionally connected to many columns to give a
    ragged row-length mix.  Diagonal = sum |off-diagonals| + shift.
    """
    rng = np.random.default_rng(seed)
    npairs = int(avg_offdiag * n / 2)
    i = rng.integers(0, n, npairs) if n > 0 else np.zeros(0, np.int64)
    j = rng.integers(0, n, npairs) if n > 0 else np.zeros(0, np.int64)
    if long_rows and n > 1:
        hubs = rng.integers(0, n, long_rows)
        fan = max(1, min(n - 1, 300))
        i = np.concatenate([i, np.repeat(hubs, fan)])
        j = np.concatenate([j, rng.integers(0, n, hubs.size * fan)])
    keep = i != j
    i, j = i[keep], j[keep]
    lo, hi = np.minimum(i, j), np.maximum(i, j)
    key = np.unique(lo * max(n, 1) + hi)
    lo, hi = key // max(n, 1), key % max(n, 1)
    w = rng.uniform(0.1, 1.0, lo.size)
    rows = np.concatenate([lo, hi, np.arange(n)])
    cols = np.concatenate([hi, lo, np.arange(n)])
    offw = np.concatenate([-w, -w])
    dsum = np.zeros(n)
    np.add.at(dsum, lo, w)
    np.add.at(dsum, hi, w)
    vals = np.concatenate([offw, dsum + shift])
    order = np.lexsort((cols, rows))
    rows, cols, vals = rows[order], cols[order], vals[order]
    rp = np.zeros(n + 1, dtype=np.int64)
    np.add.at(rp, rows + 1, 1)
    rp = np.cumsum(rp).astype(np.int32)
    return CSR(n, rp, cols.astype(np.int32), vals.astype(np.float64))


@dataclass
class Workload:
    """One solve + adjoint problem (or a batch sharing one pattern)."""
    name: str
    A: CSR                                 # pattern (and values for single systems)
    b: np.ndarray                          # [n] or [B, n]
    g: np.ndarray                          # upstream gradient dL/dx, [n] or [B, n]; see g_from_x
    rtol: float
    maxit: int
    precond: int = 0                       # 0 none, 1 Jacobi
    dtype: str = "f64"
    batch: int = 0                         # 0: single system
    values_b: Optional[np.ndarray] = None  # [B, nnz] for the batched workload
    x_star: Optional[np.ndarray] = None    # manufactured solution, if any
    x_target: Optional[np.ndarray] = None  # for L = 0.5 ||x - x_t||^2 (g = x - x_t)
    meta: dict = field(default_factory=dict)


def _stencil_apply(m: int, x: np.ndarray) -> np.ndarray:
    """b = A x for the Poisson matrix, evaluated on the grid (for the manufactured solution)."""
    X = x.reshape(m, m)
    B = 4.0 * X
    B[1:, :] -= X[:-1, :]
    B[:-1, :] -= X[1:, :]
    B[:, 1:] -= X[:, :-1]
    B[:, :-1] -= X[:, 1:]
    return B.reshape(-1)


def config1(m: int = 64) -> Workload:
    """2D Poisson m=64 (n=4096, nnz=20,224), x* ~ U(-1,1) seed 0, b = A x*, CG rtol 1e-10.

    Adjoint loss L = 0.5 ||x - x_t||^2 with x_t ~ U(-1,1) seed 1, so g = x - x_t
    (g depends on the forward solution; ``x_target`` carries x_t).
    """
    A = poisson_5pt(m)
    n = m * m
    x_star = np.random.default_rng(0).uniform(-1.0, 1.0, n)
    b = _stencil_apply(m, x_star)
    x_t = np.random.default_rng(1).uniform(-1.0, 1.0, n)
    return Workload("poisson64_cg_rtol1e-10", A, b, None, 1e-10, 100000, x_star=x_star, x_target=x_t,
                    meta={"m": m})


def config2(m: int = 1000) -> Workload:
    """2D Poisson m=1000 (n=1e6, nnz=4,996,000), b ~ N(0,1) seed 0, g ~ N(0,1) seed 1, CG rtol 1e-8."""
    A = poisson_5pt(m)
    n = m * m
    b = np.random.default_rng(0).standard_normal(n)
    g = np.random.default_rng(1).standard_normal(n)
    return Workload(f"poisson{m}_cg_rtol1e-8", A, b, g, 1e-8, 100000, meta={"m": m})


def config3(m: int = 128, batch: int = 64) -> Workload:
    """Batched shared pattern: B=64 systems on one 128x128 five-point pattern, fp32.

    System s draws, from default_rng(s): 2m(m-1) edge conductivities
    ~ log-normal(0, 0.5), then b ~ U(-1,1).  A_s = L_w + 0.01 I assembled in
    float64 and rounded to float32.  Adjoint g_s ~ U(-1,1) from
    default_rng(10000 + s).  CG rtol 1e-5.
    """
    n = m * m
    vals = None
    bs, gs = [], []
    A0 = None
    for s in range(batch):
        rng = np.random.default_rng(s)
        k = rng.lognormal(0.0, 0.5, 2 * m * (m - 1))
        As = diffusion_interior(m, k, 0.01)
        if vals is None:
            A0 = As
            vals = np.empty((batch, As.nnz), dtype=np.float32)
        vals[s] = As.values.astype(np.float32)
        bs.append(rng.uniform(-1.0, 1.0, n).astype(np.float32))
        gs.append(np.random.default_rng(10000 + s).uniform(-1.0, 1.0, n).astype(np.float32))
    pattern = CSR(n, A0.row_ptr, A0.col_idx, vals[0])
    return Workload(f"diffusion{m}_batch{batch}_fp32_cg_rtol1e-5", pattern, np.stack(bs), np.stack(gs), 1e-5,
                    100000, dtype="f32", batch=batch, values_b=vals, meta={"m": m})


def config4(m: int = 4096) -> Workload:
    """Variable-coefficient diffusion m=4096 (n=16.8M, nnz=83.9M), k ~ log-normal(0, 1.0) from
    default_rng(2), Dirichlet boundary edges; b ~ N(0,1) seed 0, g ~ N(0,1) seed 1; Jacobi PCG rtol 1e-8."""
    k = np.random.default_rng(2).lognormal(0.0, 1.0, 2 * m * (m + 1))
    A = diffusion_dirichlet(m, k)
    n = m * m
    b = np.random.default_rng(0).standard_normal(n)
    g = np.random.default_rng(1).standard_normal(n)
    return Workload(f"diffusion{m}_jacobi_pcg_rtol1e-8", A, b, g, 1e-8, 1000000, precond=1, meta={"m": m})


def config5(m: int = 13000, iters: int = 1000) -> Workload:
    """2D Poisson m=13000 (n=169M, nnz=844,948,000), int64 row_ptr; b ~ N(0,1) seed 0,
    g ~ N(0,1) seed 1; 1000 fixed CG iterations (rtol 0) forward and adjoint."""
    A = poisson_5pt(m, rowptr64=True)
    n = m * m
    b = np.random.default_rng(0).standard_normal(n)
    g = np.random.default_rng(1).standard_normal(n)
    return Workload(f"poisson{m}_cg_fixed{iters}", A, b, g, 0.0, iters, meta={"m": m})


def convdiff_bicgstab(m: int = 1000) -> Workload:
    """2D convection-diffusion m=1000 (n=1e6, nnz=4,996,000; cx = 0.4, cy = 0.25, central
    differences), b ~ N(0,1) seed 0, g ~ N(0,1) seed 1; BiCGStab rtol 1e-8 forward and adjoint."""
    A = convection_diffusion(m)
    n = m * m
    b = np.random.default_rng(0).standard_normal(n)
    g = np.random.default_rng(1).standard_normal(n)
    return Workload(f"convdiff{m}_bicgstab_rtol1e-8", A, b, g, 1e-8, 100000, meta={"m": m, "method": "bicgstab"})


def small_poisson(m: int, seed: int = 0, rowptr64: bool = False) -> Workload:
    """Small Poisson problem with b, g ~ N(0,1) (parity cases spanning several tiles)."""
    A = poisson_5pt(m, rowptr64)
    rng = np.random.default_rng(seed)
    n = m * m
    return Workload(f"poisson{m}_s{seed}", A, rng.standard_normal(n), rng.standard_normal(n), 1e-10, 100000,
                    meta={"m": m})


# Descriptive names of the five benchmark systems; config1 .. config5 are short aliases.
ALIASES = {
    "poisson64": "config1",             # 64x64 Poisson, fp64, rtol 1e-10
    "poisson1000": "config2",           # 1000x1000 Poisson, fp64, rtol 1e-8
    "diffusion128_batch64": "config3",  # 64 x 128x128 interior-edge diffusion, fp32, rtol 1e-5
    "diffusion4096_jacobi": "config4",  # 4096x4096 Dirichlet diffusion, Jacobi PCG, rtol 1e-8
    "poisson13000_int64": "config5",    # 13000x13000 Poisson, int64 row_ptr, 1000 iterations
}


def canonical_name(name: str) -> str:
    return ALIASES.get(name, name)


def config_by_name(name: str, **kw) -> Workload:
    return {"config1": config1, "config2": config2, "config3": config3, "config4": config4,
            "config5": config5, "convdiff1000_bicgstab": convdiff_bicgstab}[canonical_name(name)](**kw)
