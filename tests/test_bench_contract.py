"""Host-side pieces of the benchmark that the reported numbers rest on (CPU only)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import config_by_name, canonical_name  # noqa: E402


# algorithmic bytes per CG iteration: nnz (s_v + 4) + (n + 1) s_p + V n s_v, V = 9 (11 with Jacobi)
@pytest.mark.parametrize("name,n,nnz,s_p,jac,expect", [
    ("poisson64", 4096, 20224, 4, False, 553_988),
    ("poisson1000", 1_000_000, 4_996_000, 4, False, 135_952_004),
    ("diffusion4096_jacobi", 16_777_216, 83_869_696, 4, True, 2_549_940_228),
])
def test_bytes_per_iteration(name, n, nnz, s_p, jac, expect):
    w = config_by_name(name, m=64) if name == "poisson64" else None
    if w is not None:
        assert (w.A.n, w.A.nnz) == (n, nnz)
    assert bench.b_iter(n, nnz, 8, s_p, jac) == expect


def test_bytes_per_iteration_int64_rowptr():
    # 13000 x 13000 Poisson: nnz = 5 m^2 - 4 m, 8-byte row pointers
    m = 13000
    n, nnz = m * m, 5 * m * m - 4 * m
    assert nnz == 844_948_000
    assert bench.b_iter(n, nnz, 8, 8, False) == 23_659_376_008


def test_bytes_per_batched_iteration():
    w = config_by_name("diffusion128_batch64")
    assert (w.batch, w.A.n, w.A.nnz) == (64, 16384, 81408)
    assert bench.b_iter_batched(64, 16384, 81408, 4) == 58_980_356


def test_workload_aliases():
    assert canonical_name("poisson1000") == "config2"
    assert canonical_name("config4") == "config4"
    assert config_by_name("poisson64").name == config_by_name("config1").name


def test_traffic_record_requires_matching_sources(monkeypatch, tmp_path):
    rec = {"config2": {"dram_bytes_per_iter": 1, "source": "x", "csrc_sha256": "0" * 64}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "csrc_sha256", lambda engine: "0" * 64)
    assert bench.profiled_traffic("config2")["dram_bytes_per_iter"] == 1
    monkeypatch.setattr(bench, "csrc_sha256", lambda engine: "1" * 64)
    assert bench.profiled_traffic("config2") is None



def test_eig_gradient_bytes():
    # col_idx + gradient (nnz (s_v + 4)), row pointers, one eigenvector read once
    assert bench.b_eig_grad(1_000_000, 4_996_000, 8, 4) == 4_996_000 * 12 + 1_000_001 * 4 + 8_000_000


def test_traffic_hash_covers_each_engines_kernel_sources_only(monkeypatch, tmp_path):
    # an engine's record stays valid across changes to files holding none of its kernels, and not otherwise
    csrc = tmp_path / "differentiable_sparse_iterative_gb300" / "csrc"
    csrc.mkdir(parents=True)
    names = sorted({f for fs in bench.KERNEL_SOURCES.values() for f in fs} | {"sla_eig.cu", "sla_api.cu"})
    for name in names:
        (csrc / name).write_text(name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for engine, files in bench.KERNEL_SOURCES.items():
        h0 = bench.csrc_sha256(engine)
        for name in names:
            (csrc / name).write_text(name + " changed")
            assert (bench.csrc_sha256(engine) != h0) == (name in files), (engine, name)
            (csrc / name).write_text(name)
        assert bench.csrc_sha256(engine) == h0
    assert set(bench.ENGINE_OF) == {"config1", "config2", "config3", "config4", "config5", "convdiff1000_bicgstab"}


def test_bicgstab_iteration_bytes():
    # two matrix streams (values + col_idx, row pointers) and 17 vector passes of 8 bytes per row
    n, nnz = 1_000_000, 4_996_000
    assert bench.b_iter_bicgstab(n, nnz, 8, 4) == 2 * (nnz * 12 + (n + 1) * 4) + 17 * n * 8
    # 2 nnz flops per product, two products, and 12 multiply-adds per row
    assert bench.flops_iter_bicgstab(n, nnz) == 2 * 2 * nnz + 2 * 12 * n
